// capi.cu -- the extern "C" boundary declared in include/conv_bn_silu.h:
// argument validation, output sizes, kernel choice and launch, error words.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "conv_bn_silu.h"
#include "cbs_internal.h"

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    return CBS_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int dims_from(int h, int w_in, int r, int s, int sh, int sw, int ph, int pw, int *ho, int *wo)
{
    if (h < 1 || w_in < 1 || r < 1 || s < 1 || sh < 1 || sw < 1 || ph < 0 || pw < 0)
        return CBS_ERR_INVALID_ARG;
    const long long hp = (long long)h + 2LL * ph, wp = (long long)w_in + 2LL * pw;
    if (hp < r || wp < s) return CBS_ERR_INVALID_ARG;
    const long long oh = (hp - r) / sh + 1, ow = (wp - s) / sw + 1;
    if (oh < 1 || ow < 1 || oh > 0x7fffffffLL || ow > 0x7fffffffLL) return CBS_ERR_INVALID_ARG;
    *ho = (int)oh;
    *wo = (int)ow;
    return CBS_OK;
}

// Shape checks shared by forward and plan.  Fills everything but the pointers.
int make_problem(int n, int h, int w_in, int c, int c_out, int r, int s, int sh, int sw, int ph, int pw,
                 cbs::ConvProblem *p)
{
    if (n < 0 || c < 1 || c_out < 0) return CBS_ERR_INVALID_ARG;
    int ho = 0, wo = 0;
    const int st = dims_from(h, w_in, r, s, sh, sw, ph, pw, &ho, &wo);
    if (st != CBS_OK) return st;
    p->n = n;
    p->h = h;
    p->w_in = w_in;
    p->c = c;
    p->c_out = c_out;
    p->r = r;
    p->s = s;
    p->stride_h = sh;
    p->stride_w = sw;
    p->pad_h = ph;
    p->pad_w = pw;
    p->ho = ho;
    p->wo = wo;
    p->m = (long long)n * ho * wo;
    // Keep every tensor's element count within 2^62 so byte offsets never overflow.
    const long long xe = (long long)n * h * w_in;
    if (xe > (1LL << 40) / (c > 0 ? c : 1) || p->m > (1LL << 40) / (c_out > 0 ? c_out : 1) ||
        (long long)r * s * c > (1LL << 31) - 1)
        return CBS_ERR_INVALID_ARG;
    return CBS_OK;
}

int select_algo(const cbs::ConvProblem &p, int algo)
{
    if (algo != CBS_ALGO_AUTO) return algo;
    return cbs::tc_supported(p) || cbs::gather_supported(p) ? CBS_ALGO_TCGEN05 : CBS_ALGO_DIRECT;
}

int sm_count_current_device(int *count)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    static std::mutex mu;
    static std::vector<int> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        if ((int)cache.size() > dev && cache[dev] > 0) {
            *count = cache[dev];
            return CBS_OK;
        }
    }
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1, 0);
    cache[dev] = v;
    *count = v;
    return CBS_OK;
}

// A request's tcgen05 overrides, or nullptr when it leaves every choice to the planner.
bool has_overrides(const cbs::PlanRequest *rq)
{
    return rq && (rq->swap_ab >= 0 || rq->stream_k >= 0 || rq->pair >= 0 || rq->block_n != 0 ||
                  rq->balanced >= 0 || rq->wres >= 0 || rq->row_boxes >= 0);
}

// Validated problem (pointers set) -> the chosen kernel's launch on `strm`.
int launch_forward(const cbs::ConvProblem &p, int algo, cudaStream_t strm, const cbs::PlanRequest *rq = nullptr)
{
    const int chosen = select_algo(p, algo);
    if (chosen == CBS_ALGO_TCGEN05) {
        if (!cbs::tc_supported(p) && !cbs::gather_supported(p)) return CBS_ERR_UNSUPPORTED;
        int sms = 0;
        const int st = sm_count_current_device(&sms);
        if (st != CBS_OK) return st;
        if (!cbs::tc_supported(p)) {
            if (has_overrides(rq)) return CBS_ERR_UNSUPPORTED;  // the thin-input kernel has no such choices
            cudaError_t e = cbs::gather_launch(p, sms, strm);
            return e == cudaSuccess ? CBS_OK : cuda_fail(e);
        }
        cbs::TcPlan plan{};
        if (cbs::tc_make_plan_request(p, sms, rq, &plan) != 0) return CBS_ERR_UNSUPPORTED;
        // A stream-K plan needs the library-held workspace of this (device, stream).
        if (plan.stream_k && !cbs::tc_workspace_reserve(strm)) return CBS_ERR_UNSUPPORTED;
        cudaError_t e = cbs::tc_launch(p, plan, strm);
        return e == cudaSuccess ? CBS_OK : cuda_fail(e);
    }
    if (has_overrides(rq)) return CBS_ERR_UNSUPPORTED;
    cudaError_t e = cbs::direct_launch(p, strm);
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

// cbs_plan_request -> checked algorithm and planner overrides.
int read_request(const cbs_plan_request *req, int *algo, cbs::PlanRequest *rq)
{
    if (!req) return CBS_ERR_INVALID_ARG;
    if (req->wait_timeout_ns < 0) return CBS_ERR_INVALID_ARG;
    if (req->algo < CBS_ALGO_AUTO || req->algo > CBS_ALGO_DIRECT) return CBS_ERR_INVALID_ARG;
    for (int v : {req->swap_ab, req->stream_k, req->pair, req->balanced, req->weights_resident, req->row_boxes})
        if (v < -1 || v > 1) return CBS_ERR_INVALID_ARG;
    if (req->block_n != 0 && req->block_n != 16 && req->block_n != 32 && req->block_n != 64 &&
        req->block_n != 128 && req->block_n != 256)
        return CBS_ERR_INVALID_ARG;
    *algo = req->algo;
    *rq = cbs::PlanRequest{req->swap_ab, req->stream_k, req->pair, req->block_n, req->balanced,
                           req->weights_resident, req->row_boxes};
    return CBS_OK;
}

// ------------------------------------------------------------------ allocation-free forward
// Scratch for conv_bn_silu_forward_noalloc: the stream-K partial tiles and ready
// flags live in this fixed device array instead of library-allocated memory.
// It is zero-initialised when the module loads; every GPU that loads the
// library holds it until the process exits.  In host code the symbol is only a
// stand-in: its device address comes from cudaGetSymbolAddress below.
constexpr size_t kNoAllocScratchBytes = 20u << 20;  // 20 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device (on that device's first call) and cached.
int noalloc_scratch_address(void **out)
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64) return CBS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e);
        addr[dev] = p;
    }
    *out = addr[dev];
    return CBS_OK;
}

}  // namespace

extern "C" {

int conv_bn_silu_forward_noalloc(const void *x, const void *w, const float *scale, const float *bias,
                                 void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                                 int stride_h, int stride_w, int pad_h, int pad_w, void *stream)
{
    cbs::ConvProblem p{};
    int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(y))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = y;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    // Set-up, on the first call on each device: the scratch array's device address.
    void *scratch = nullptr;
    st = noalloc_scratch_address(&scratch);
    if (st != CBS_OK) return st;
    int sms = 0;
    if (!cbs::tc_supported(p)) {  // neither of these kernels needs scratch
        cudaError_t e;
        if (cbs::gather_supported(p)) {
            st = sm_count_current_device(&sms);
            if (st != CBS_OK) return st;
            e = cbs::gather_launch(p, sms, strm);
        } else {
            e = cbs::direct_launch(p, strm);
        }
        return e == cudaSuccess ? CBS_OK : cuda_fail(e);
    }
    st = sm_count_current_device(&sms);
    if (st != CBS_OK) return st;
    cbs::TcPlan plan = cbs::tc_make_plan(p, sms);
    if (plan.stream_k && plan.workspace_bytes > (long long)kNoAllocScratchBytes) {
        // The split would not fit the array (a GPU with many more SMs than GB300's 152):
        // whole tiles per CTA instead, which need no scratch.
        const cbs::PlanRequest whole{-1, 0, 0, 0, -1, -1, -1};
        if (cbs::tc_make_plan_request(p, sms, &whole, &plan) != 0) return CBS_ERR_UNSUPPORTED;
    }
    if (plan.stream_k) {
        // The ready flags must start at zero; a previous call that gave up may have left some set.
        cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)plan.flag_bytes, strm);
        if (e != cudaSuccess) return cuda_fail(e);
    } else {
        scratch = nullptr;
    }
    cudaError_t e = cbs::tc_launch_with_workspace(p, plan, strm, scratch);
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_fold(const float *gamma, const float *beta, const float *mean, const float *var,
                      float eps, int c_out, float *scale, float *bias, void *stream)
{
    if (c_out < 0 || !(eps >= 0.0f) || eps > 3.0e38f) return CBS_ERR_INVALID_ARG;
    if (c_out == 0) return CBS_OK;
    if (!gamma || !beta || !mean || !var || !scale || !bias) return CBS_ERR_INVALID_ARG;
    if (!aligned16(gamma) || !aligned16(beta) || !aligned16(mean) || !aligned16(var) ||
        !aligned16(scale) || !aligned16(bias))
        return CBS_ERR_MISALIGNED;
    cudaError_t e = cbs::fold_launch(gamma, beta, mean, var, eps, c_out, scale, bias,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_fold_batch(const cbs_fold_layer *layers, int n_layers, void *stream)
{
    if (n_layers < 0 || (n_layers > 0 && !layers)) return CBS_ERR_INVALID_ARG;
    std::vector<cbs::FoldLayer> v;
    v.reserve((size_t)n_layers);
    for (int i = 0; i < n_layers; ++i) {
        const cbs_fold_layer &L = layers[i];
        if (L.c_out < 0 || !(L.eps >= 0.0f) || L.eps > 3.0e38f) return CBS_ERR_INVALID_ARG;
        if (L.c_out == 0) continue;
        if (!L.gamma || !L.beta || !L.mean || !L.var || !L.scale || !L.bias) return CBS_ERR_INVALID_ARG;
        if (!aligned16(L.gamma) || !aligned16(L.beta) || !aligned16(L.mean) || !aligned16(L.var) ||
            !aligned16(L.scale) || !aligned16(L.bias))
            return CBS_ERR_MISALIGNED;
        v.push_back(cbs::FoldLayer{L.gamma, L.beta, L.mean, L.var, L.eps, L.c_out, L.scale, L.bias});
    }
    if (v.empty()) return CBS_OK;
    cudaError_t e = cbs::fold_batch_launch(v.data(), (int)v.size(), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_forward_algo(const void *x, const void *w, const float *scale, const float *bias,
                              void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                              int stride_h, int stride_w, int pad_h, int pad_w, int algo, void *stream)
{
    if (algo < CBS_ALGO_AUTO || algo > CBS_ALGO_DIRECT) return CBS_ERR_INVALID_ARG;
    cbs::ConvProblem p{};
    int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(y))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = y;
    return launch_forward(p, algo, static_cast<cudaStream_t>(stream));
}

int conv_bn_act_forward(const void *x, const void *w, const float *scale, const float *bias,
                        const void *residual, void *y, int n, int h, int w_in, int c, int c_out, int r,
                        int s, int stride_h, int stride_w, int pad_h, int pad_w, int activation,
                        void *stream)
{
    int mode;
    switch (activation) {
    case CBS_ACT_SILU: mode = cbs::kEpiSilu; break;
    case CBS_ACT_IDENTITY: mode = cbs::kEpiBn; break;
    case CBS_ACT_RELU: mode = cbs::kEpiRelu; break;
    default: return CBS_ERR_INVALID_ARG;
    }
    cbs::ConvProblem p{};
    int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(y) ||
        (residual && !aligned16(residual)))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = y;
    p.epi_mode = mode;
    p.residual = residual;
    return launch_forward(p, CBS_ALGO_AUTO, static_cast<cudaStream_t>(stream));
}

int conv_bn_act_forward_fp8(const void *x, const void *w, const float *scale, const float *bias, void *y,
                            int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h, int stride_w,
                            int pad_h, int pad_w, int activation, void *stream)
{
    int mode;
    switch (activation) {
    case CBS_ACT_SILU: mode = cbs::kEpiSilu; break;
    case CBS_ACT_IDENTITY: mode = cbs::kEpiBn; break;
    case CBS_ACT_RELU: mode = cbs::kEpiRelu; break;
    default: return CBS_ERR_INVALID_ARG;
    }
    cbs::ConvProblem p{};
    int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(y))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = y;
    p.epi_mode = mode;
    p.out_fp8 = 1;
    return launch_forward(p, CBS_ALGO_AUTO, static_cast<cudaStream_t>(stream));
}

int conv_bn_silu_forward_unfused(const void *x, const void *w, const float *scale, const float *bias,
                                 void *t1, void *t2, void *y, int n, int h, int w_in, int c, int c_out,
                                 int r, int s, int stride_h, int stride_w, int pad_h, int pad_w,
                                 void *stream)
{
    cbs::ConvProblem p{};
    int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !t1 || !t2 || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(t1) ||
        !aligned16(t2) || !aligned16(y))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = t1;
    p.epi_mode = cbs::kEpiConvOnly;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    st = launch_forward(p, CBS_ALGO_AUTO, strm);
    if (st != CBS_OK) return st;
    const long long count = p.m * c_out;
    cudaError_t e = cbs::bn_apply_launch(t1, scale, bias, t2, count, c_out, strm);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cbs::silu_apply_launch(t2, y, count, strm);
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_bn_apply(const void *t1, const float *scale, const float *bias, void *t2,
                          long long count, int c_out, void *stream)
{
    if (count < 0 || c_out < 1 || count % c_out != 0) return CBS_ERR_INVALID_ARG;
    if (count > (1LL << 40)) return CBS_ERR_INVALID_ARG;
    if (count == 0) return CBS_OK;
    if (!t1 || !scale || !bias || !t2) return CBS_ERR_INVALID_ARG;
    if (!aligned16(t1) || !aligned16(scale) || !aligned16(bias) || !aligned16(t2)) return CBS_ERR_MISALIGNED;
    cudaError_t e = cbs::bn_apply_launch(t1, scale, bias, t2, count, c_out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_silu_apply(const void *t2, void *y, long long count, void *stream)
{
    if (count < 0 || count > (1LL << 40)) return CBS_ERR_INVALID_ARG;
    if (count == 0) return CBS_OK;
    if (!t2 || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(t2) || !aligned16(y)) return CBS_ERR_MISALIGNED;
    cudaError_t e = cbs::silu_apply_launch(t2, y, count, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CBS_OK : cuda_fail(e);
}

int conv_bn_silu_forward(const void *x, const void *w, const float *scale, const float *bias, void *y,
                         int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h,
                         int stride_w, int pad_h, int pad_w, void *stream)
{
    return conv_bn_silu_forward_algo(x, w, scale, bias, y, n, h, w_in, c, c_out, r, s, stride_h,
                                     stride_w, pad_h, pad_w, CBS_ALGO_AUTO, stream);
}

int conv_bn_silu_output_dims(int h, int w_in, int r, int s, int stride_h, int stride_w, int pad_h,
                             int pad_w, int *ho, int *wo)
{
    if (!ho || !wo) return CBS_ERR_INVALID_ARG;
    return dims_from(h, w_in, r, s, stride_h, stride_w, pad_h, pad_w, ho, wo);
}

static int fill_plan(const cbs::ConvProblem &p, int algo, int sm_count, const cbs::PlanRequest *rq,
                     cbs_plan_info *info)
{
    const int n = p.n, c = p.c, c_out = p.c_out, r = p.r, s = p.s;
    (void)n;
    const int chosen = select_algo(p, algo);
    cbs_plan_info out{};
    out.algo = chosen;
    if (chosen == CBS_ALGO_TCGEN05 && !cbs::tc_supported(p)) {
        // Thin-input kernel: 128-pixel tiles, K zero-padded to 32 or 64, each CTA an equal
        // range of pixels whose input rows it stages in shared memory.
        cbs::GatherPlan g{};
        if (has_overrides(rq) || !cbs::gather_plan(p, sm_count, &g)) return CBS_ERR_UNSUPPORTED;
        out.block_m = 128;
        out.block_n = g.block_n;
        out.block_k = g.block_k;
        out.stages = g.stages;
        out.tiles = g.tiles;
        out.grid = g.grid;
        out.threads = cbs::kGatherBlockThreads;
        out.smem_bytes = g.smem_bytes;
        out.k_iters = 1;
        out.cluster = 1;
    } else if (chosen == CBS_ALGO_TCGEN05) {
        cbs::TcPlan t{};
        if (cbs::tc_make_plan_request(p, sm_count, rq, &t) != 0) return CBS_ERR_UNSUPPORTED;
        out.block_m = t.cmajor ? t.cm_unit_px : (t.swap_ab ? t.block_n : cbs::kTcBlockM);  // output pixels per tile
        out.block_n = t.swap_ab ? cbs::kTcBlockM : t.block_n;  // output channels per tile
        out.block_k = t.block_k;
        out.stages = t.stages;
        out.tiles = t.m_tiles * t.n_tiles;
        out.grid = t.grid;
        out.threads = t.cmajor ? cbs::kCmThreads : cbs::tc_threads(t.block_n, t.pair != 0);
        out.smem_bytes = t.smem_bytes;
        out.k_iters = t.k_iters;
        out.stream_k = t.stream_k;
        out.swap_ab = t.swap_ab;
        out.cluster = t.pair ? 2 : 1;
        out.workspace_bytes = t.workspace_bytes;
        out.balanced = t.balanced;
        out.weights_resident = t.cmajor ? t.cm_wres : 0;
        out.row_boxes = t.cmajor && t.cm_xmode != 0 ? 1 : 0;
    } else {
        if (has_overrides(rq)) return CBS_ERR_UNSUPPORTED;  // the direct kernel has no tilings to choose
        const long long bx = (p.m + cbs::kDirectThreads - 1) / cbs::kDirectThreads;
        const int by = (c_out + cbs::kDirectBlockN - 1) / cbs::kDirectBlockN;
        out.block_m = cbs::kDirectThreads;
        out.block_n = cbs::kDirectBlockN;
        out.block_k = 1;
        out.stages = 0;
        out.tiles = (int)(bx * by);
        out.grid = out.tiles;
        out.threads = cbs::kDirectThreads;
        out.smem_bytes = 0;
        out.k_iters = r * s * c;
    }
    *info = out;
    return CBS_OK;
}

int conv_bn_silu_plan(int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h, int stride_w,
                      int pad_h, int pad_w, int algo, int sm_count, cbs_plan_info *info)
{
    if (!info || sm_count < 1 || algo < CBS_ALGO_AUTO || algo > CBS_ALGO_DIRECT)
        return CBS_ERR_INVALID_ARG;
    cbs::ConvProblem p{};
    const int st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    return fill_plan(p, algo, sm_count, nullptr, info);
}

int conv_bn_silu_plan_request(int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h,
                              int stride_w, int pad_h, int pad_w, const cbs_plan_request *req, int sm_count,
                              cbs_plan_info *info)
{
    if (!info || sm_count < 1) return CBS_ERR_INVALID_ARG;
    int algo = 0;
    cbs::PlanRequest rq{};
    int st = read_request(req, &algo, &rq);
    if (st != CBS_OK) return st;
    cbs::ConvProblem p{};
    st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    return fill_plan(p, algo, sm_count, &rq, info);
}

int conv_bn_silu_forward_request(const void *x, const void *w, const float *scale, const float *bias,
                                 void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                                 int stride_h, int stride_w, int pad_h, int pad_w, const cbs_plan_request *req,
                                 void *stream)
{
    int algo = 0;
    cbs::PlanRequest rq{};
    int st = read_request(req, &algo, &rq);
    if (st != CBS_OK) return st;
    cbs::ConvProblem p{};
    st = make_problem(n, h, w_in, c, c_out, r, s, stride_h, stride_w, pad_h, pad_w, &p);
    if (st != CBS_OK) return st;
    if (p.m == 0 || c_out == 0) return CBS_OK;
    if (!x || !w || !scale || !bias || !y) return CBS_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(scale) || !aligned16(bias) || !aligned16(y))
        return CBS_ERR_MISALIGNED;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.bias = bias;
    p.y = y;
    p.wait_timeout_ns = req->wait_timeout_ns;
    return launch_forward(p, algo, static_cast<cudaStream_t>(stream), &rq);
}

int conv_bn_silu_check(void *stream)
{
    unsigned int word = 0;
    cudaError_t e = cbs::tc_read_and_clear_error(static_cast<cudaStream_t>(stream), &word);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int gword = 0;
    e = cbs::gather_read_and_clear_error(static_cast<cudaStream_t>(stream), &gword);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int wword = 0;
    e = cbs::cmajor_read_and_clear_error(static_cast<cudaStream_t>(stream), &wword);
    if (e != cudaSuccess) return cuda_fail(e);
    if ((gword != 0 || wword != 0) && word == 0) return CBS_ERR_TIMEOUT;
    if (word == 0) return CBS_OK;
    // A kernel gave up mid-way: stream-K ready flags may be left raised.
    e = cbs::tc_reset_workspaces();
    if (e != cudaSuccess) return cuda_fail(e);
    return CBS_ERR_TIMEOUT;
}

const char *conv_bn_silu_status_string(int status)
{
    switch (status) {
    case CBS_OK: return "ok";
    case CBS_ERR_INVALID_ARG: return "invalid argument";
    case CBS_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case CBS_ERR_UNSUPPORTED: return "shape not supported by the requested kernel";
    case CBS_ERR_CUDA: return "CUDA error";
    case CBS_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    default: return "unknown status";
    }
}

int conv_bn_silu_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"
