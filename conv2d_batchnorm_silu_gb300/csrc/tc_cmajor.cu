// tc_cmajor.cu -- fused conv2d + BatchNorm + SiLU on channel-major ("swap AB")
// tiles, built for the layers that are bound by moving x and y.
//
// GEMM view as in tc_conv.cu, transposed: D[channel][pixel] = W[channel][k] *
// X[pixel][k]^T, K laid out (r, s, c) and visited in K steps of one tap x BK
// channels, the taps running fastest; a CTA owns one 128-channel tile and a
// sequence of pixel units.  Two choices are template switches, picked per
// shape by the planner:
//   - XMODE: how x reaches shared memory.  kXIm2col: one im2col box per K step
//     (a run of output pixels of one filter tap).  kXRows: a unit is a group of
//     whole output rows of one image, and each K step's operand is one tiled
//     box of x viewed as (stride*C, W/stride, H, N): output pixel ow of tap s
//     reads input pixel stride*ow - pad + s, which in that view is element
//     (s - pad) mod stride of "pixel" ow + floor((s - pad) / stride), and the
//     box walks the unit's input rows with a traversal stride of `stride`.
//     kXMatrix (1x1, stride 1, no padding): x is the [M][C] matrix itself and
//     each K step's operand one tiled box of its rows.  On GB300 the TMA unit
//     moves tiled boxes at about 1.5x the rate of im2col boxes.
//   - WRES: where the weights live.  On: each CTA copies its 128-channel weight
//     tile into tensor memory once (TMA into a stage, then tcgen05.cp) and the
//     MMAs read their A operand from there; only x streams.  Off: one 128 x BK
//     weight load per K step next to the x box, the MMAs read both operands
//     from shared memory, and the accumulators may use all of tensor memory.
// Warp roles: warp 0 TMA producer of x, warp 2 of the weights, warp 1 MMA issuer
// (one thread), warps 4..15 epilogue (BN multiply/add, activation, bf16, transposed
// to NHWC through shared memory, TMA stores of 32 channels x 16 pixels; three warps
// per TMEM lane quarter, since with two the epilogue, not the K loop, set the pace).  Accumulators are
// double buffered in TMEM, so the epilogue of one unit runs under the K loop of
// the next.  Every wait is bounded in time; on a timeout the kernel records an
// error bit, waits for its own copies in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {

__device__ unsigned int g_cmajor_error = 0;

namespace {

constexpr uint64_t kCmTimeoutNs = 2000000000ull;
constexpr int kCmMaxStages = 16;
constexpr int kCmChunk = 16;            // pixels per epilogue chunk (one TMA store of 32 channels)
constexpr int kCmStgBytes = kCmChunk * 32 * 2;
constexpr int kCmSmemLimit = 232448;
constexpr int kEpiCmSilu = 0;           // the fused layer's own epilogue
constexpr int kEpiCmMode = 1;           // the launch's EpiMode, chosen at run time
constexpr int kXIm2col = 0, kXRows = 1, kXMatrix = 2;  // how x is loaded (see above)

struct CmArgs {
    const float *scale;
    const float *bias;
    int c, c_out, m;
    int ho, wo, howo, stride_h, stride_w, pad_h, pad_w, s;
    int c_chunks, k_iters;
    int ctas_per_tile;   // CTAs sharing one 128-channel tile; the grid is ctas_per_tile x channel tiles
    int unit_px;         // pixels per unit (im2col box), or rows * wo (row boxes); a multiple of 16
    int unit_rows;       // row boxes: output rows per unit
    int groups;          // row boxes: row groups per image, ceil(ho / unit_rows)
    int stages, stage_bytes, a_bytes;  // a_bytes: the weight part of a stage (streamed weights)
    int epi_mode;
    unsigned long long wait_ns;
};

__device__ __forceinline__ void cm_error(unsigned int bit, volatile int *abort_flag)
{
    atomicOr(&g_cmajor_error, bit);
    *abort_flag = 1;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulate, shape from idesc.
__device__ __forceinline__ void mma_tmem_a(uint32_t d, uint32_t a, uint64_t b_desc, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// 128 rows x 32 bytes (one K = 16 slab of a 128-row bf16 tile) from shared memory,
// described like an MMA operand, into TMEM lanes 0..127, 8 columns from `taddr`.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t s_desc)
{
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(s_desc) : "memory");
}

// Tiled 2-D load (x as the [M][C] matrix of a 1x1 layer), completion on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d_rows(uint32_t dst, const CUtensorMap *tm, uint32_t bar, int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Tiled 4-D load (the row-box view of x), completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *tm, uint32_t bar, int c0, int c1,
                                            int c2, int c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// The units one CTA processes, in order.  Pixel units (im2col or matrix boxes): the
// CTA's equal share of the pixels, in whole 16-pixel chunks (so no epilogue store of 16
// pixels crosses into another CTA's share), cut into runs of unit_px.  Row units (row
// boxes): the (image, row group) units, dealt round-robin over the tile's CTAs.
struct CmUnit {
    int p0, np;      // first output pixel and pixel count
    int img, oh0;    // row units: image and first output row
};

template <int XMODE>
struct CmIter {
    static constexpr bool XROWS = XMODE == kXRows;
    int next, end, step;
    __device__ CmIter(const CmArgs &a, int j)
    {
        if constexpr (XROWS) {
            next = j;
            end = (a.m / a.howo) * a.groups;  // images x row groups
            step = a.ctas_per_tile;
        } else {
            const int chunks = (a.m + kCmChunk - 1) / kCmChunk;
            const int base = chunks / a.ctas_per_tile, extra = chunks - base * a.ctas_per_tile;
            const int c0 = j * base + (j < extra ? j : extra);
            const int c1 = c0 + base + (j < extra ? 1 : 0);
            next = c0 * kCmChunk;
            end = c1 * kCmChunk < a.m ? c1 * kCmChunk : a.m;
            step = a.unit_px;
        }
    }
    __device__ bool get(const CmArgs &a, CmUnit &u)
    {
        if (next >= end) return false;
        if constexpr (XROWS) {
            u.img = next / a.groups;
            const int g = next - u.img * a.groups;
            u.oh0 = g * a.unit_rows;
            const int rows = a.ho - u.oh0 < a.unit_rows ? a.ho - u.oh0 : a.unit_rows;
            u.p0 = u.img * a.howo + u.oh0 * a.wo;
            u.np = rows * a.wo;
        } else {
            u.p0 = next;
            u.np = end - next < a.unit_px ? end - next : a.unit_px;
            u.img = u.oh0 = 0;
        }
        next += step;
        return true;
    }
};

template <int BK, int EPI, bool WRES, int XMODE>
__global__ void __launch_bounds__(kCmThreads, 1)
    tc_cmajor_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_y, const CmArgs a)
{
    constexpr int ROW = BK * 2;  // operand row bytes = swizzle span
    const int emode = EPI == kEpiCmSilu ? (int)kEpiSilu : a.epi_mode;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sm_stage = smem;
    uint8_t *sm_stg = sm_stage + a.stages * a.stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_stg + kCmEpiWarps * 2 * kCmStgBytes);
    uint64_t *full = bars;
    uint64_t *empty = full + kCmMaxStages;
    uint64_t *tfull = empty + kCmMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *wready = tempty + 2;  // resident weights: the weights are in TMEM
    uint64_t *drain = wready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ct = (int)blockIdx.x / a.ctas_per_tile;  // this CTA's 128-channel tile
    const int jcta = (int)blockIdx.x - ct * a.ctas_per_tile;
    const int wcols = WRES ? a.k_iters * (BK / 2) : 0;  // TMEM columns holding the weights
    // The x operand's bytes in a stage (streamed weights: after the weight part).
    const int b_off = WRES ? 0 : a.a_bytes;

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            dev::mbar_init(dev::smem_u32(&full[i]), WRES ? 1 : 2);  // one arrival per producer
            dev::mbar_init(dev::smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&tfull[i]), 1);
            dev::mbar_init(dev::smem_u32(&tempty[i]), kCmEpiWarps);
        }
        dev::mbar_init(dev::smem_u32(wready), 1);
        dev::mbar_init(dev::smem_u32(drain), 1);
        *abort_flag = 0;
        dev::fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        dev::prefetch_tensormap(&tm_x);
        dev::prefetch_tensormap(&tm_w);
        dev::prefetch_tensormap(&tm_y);
    }
    if (warp == 1) {
        dev::tmem_alloc<1>(dev::smem_u32(tmem_slot), 512);
        dev::tmem_relinquish_alloc_permit<1>();
    }
    dev::tc_fence_before_sync();
    __syncthreads();
    dev::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();

    if (warp == 0 || (!WRES && warp == 2)) {
        // ------------------------------------------------------------ producers
        // Streamed weights: warp 0 loads the x boxes and warp 2 the weight tiles, each
        // arriving on the stage's full barrier with its own byte count (two issuing threads
        // keep more of the load path busy than one).  Resident weights: warp 0 alone.
        const bool loads_w = warp == 2;
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            bool ok = true;
            auto next_stage = [&]() {
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            auto wait_empty = [&]() {
                if (!dev::mbar_wait_bounded(dev::smem_u32(&empty[stage]), phase ^ 1u, abort_flag, a.wait_ns)) {
                    if (!*abort_flag) cm_error(kErrTimeoutProducer, abort_flag);
                    return false;
                }
                return true;
            };
            auto mark_issued = [&]() {
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            };
            // K step it reads filter tap it % taps of channel chunk it / taps: the taps run
            // fastest, so a unit's first steps read one chunk of its input rows, not all of them.
            const int taps = a.k_iters / a.c_chunks;
            if constexpr (WRES) {
                // The resident weight tile first: one load of 128 channels x BK per K step,
                // in the K order of the MMAs.
                for (int it = 0; it < a.k_iters && ok; ++it) {
                    if (!(ok = wait_empty())) break;
                    const uint32_t f_bar = dev::smem_u32(&full[stage]);
                    dev::mbar_arrive_expect_tx(f_bar, 128 * BK * 2);
                    const int cc = it / taps, tap = it - cc * taps;
                    dev::tma_load_3d(dev::smem_u32(sm_stage + stage * a.stage_bytes), &tm_w, f_bar, cc * BK, tap,
                                     ct * 128);
                    mark_issued();
                    next_stage();
                }
            }
            CmIter<XMODE> iter(a, jcta);
            CmUnit u;
            const uint32_t x_bytes = (uint32_t)(a.unit_px * BK * 2);
            while (ok && !*abort_flag && iter.get(a, u)) {
                int corner_w = 0, corner_h = 0, img = 0;
                if constexpr (XMODE == kXIm2col) {
                    img = u.p0 / a.howo;
                    const int rem = u.p0 - img * a.howo;
                    const int oh = rem / a.wo;
                    const int ow = rem - oh * a.wo;
                    corner_w = ow * a.stride_w - a.pad_w;
                    corner_h = oh * a.stride_h - a.pad_h;
                }
                int cc = 0, s = 0, r = 0;
                for (int it = 0; it < a.k_iters; ++it) {
                    if (!(ok = wait_empty())) break;
                    const uint32_t f_bar = dev::smem_u32(&full[stage]);
                    const uint32_t dst = dev::smem_u32(sm_stage + stage * a.stage_bytes);
                    if (loads_w) {
                        dev::mbar_arrive_expect_tx(f_bar, 128u * BK * 2u);
                        dev::tma_load_3d(dst, &tm_w, f_bar, cc * BK, r * a.s + s, ct * 128);
                    } else if constexpr (XMODE == kXMatrix) {
                        dev::mbar_arrive_expect_tx(f_bar, x_bytes);
                        tma_load_2d_rows(dst + (uint32_t)b_off, &tm_x, f_bar, cc * BK, u.p0);
                    } else if constexpr (XMODE == kXRows) {
                        dev::mbar_arrive_expect_tx(f_bar, x_bytes);
                        // Input pixel stride*ow - pad + s of row stride*oh - pad + r: in the
                        // (stride*C, W/stride, H, N) view, element (s - pad) mod stride of
                        // "pixel" ow + floor((s - pad) / stride).
                        const int d = s - a.pad_w;
                        const int q = d >= 0 ? d / a.stride_w : -((-d + a.stride_w - 1) / a.stride_w);
                        const int half = d - q * a.stride_w;
                        tma_load_4d(dst + (uint32_t)b_off, &tm_x, f_bar, half * a.c + cc * BK, q,
                                    u.oh0 * a.stride_h - a.pad_h + r, u.img);
                    } else {
                        dev::mbar_arrive_expect_tx(f_bar, x_bytes);
                        dev::tma_load_im2col_4d(dst + (uint32_t)b_off, &tm_x, f_bar, cc * BK, corner_w, corner_h, img,
                                                (uint16_t)s, (uint16_t)r);
                    }
                    mark_issued();
                    if (++s == a.s) {
                        s = 0;
                        if (++r * a.s == taps) {
                            r = 0;
                            ++cc;
                        }
                    }
                    next_stage();
                }
            }
            // Every load issued must land before the CTA may exit (one bounded drain wait).
            bool drain_ok = true;
            for (int i = 0; i < a.stages && drain_ok; ++i)
                if ((issued >> i) & 1u)
                    if (!dev::mbar_wait_bounded(dev::smem_u32(&full[i]), (issued_parity >> i) & 1u, nullptr,
                                                kCmTimeoutNs)) {
                        cm_error(kErrTimeoutDrain, abort_flag);
                        drain_ok = false;
                    }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            auto next_stage = [&]() {
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            };
            if constexpr (WRES) {
                // The weight tile into TMEM columns [0, wcols): K step it, slab kk of 16
                // channels, goes to columns it*BK/2 + kk*8 (two bf16 per 32-bit column).
                for (int it = 0; it < a.k_iters; ++it) {
                    if (!dev::mbar_wait_bounded(dev::smem_u32(&full[stage]), phase, abort_flag, a.wait_ns)) {
                        if (!*abort_flag) cm_error(kErrTimeoutMma, abort_flag);
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after_sync();
                    const uint64_t ds = dev::smem_desc_kmajor(dev::smem_u32(sm_stage + stage * a.stage_bytes), ROW);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tmem_cp_128x256b(tmem_base + (uint32_t)(it * (BK / 2) + kk * 8), ds + (uint64_t)(2 * kk));
                    dev::tc_commit<1>(dev::smem_u32(&empty[stage]));
                    next_stage();
                }
                if (ok) {
                    dev::tc_commit<1>(dev::smem_u32(wready));
                    if (!dev::mbar_wait_bounded(dev::smem_u32(wready), 0, abort_flag, a.wait_ns)) {
                        if (!*abort_flag) cm_error(kErrTimeoutMma, abort_flag);
                        ok = false;
                    }
                }
            }
            CmIter<XMODE> iter(a, jcta);
            CmUnit u;
            int lt = 0;
            for (; ok && iter.get(a, u); ++lt) {
                const int buf = lt & 1;
                const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
                if (!dev::mbar_wait_bounded(dev::smem_u32(&tempty[buf]), tparity ^ 1u, abort_flag, a.wait_ns)) {
                    if (!*abort_flag) cm_error(kErrTimeoutMma, abort_flag);
                    break;
                }
                dev::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(wcols + buf * a.unit_px);
                // The MMA's N is the unit's pixel count rounded up to 16 (the rows past it are
                // loaded neighbours or zeros and are never stored).
                const uint32_t idesc = dev::idesc_bf16_f32(128, (u.np + 15) & ~15);
                for (int it = 0; it < a.k_iters; ++it) {
                    if (!dev::mbar_wait_bounded(dev::smem_u32(&full[stage]), phase, abort_flag, a.wait_ns)) {
                        if (!*abort_flag) cm_error(kErrTimeoutMma, abort_flag);
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after_sync();
                    const uint32_t st = dev::smem_u32(sm_stage + stage * a.stage_bytes);
                    const uint64_t db = dev::smem_desc_kmajor(st + (uint32_t)b_off, ROW);
                    if constexpr (WRES) {
                        const uint32_t wa = tmem_base + (uint32_t)(it * (BK / 2));
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            mma_tmem_a(d_tmem, wa + (uint32_t)(kk * 8), db + (uint64_t)(2 * kk), idesc,
                                       (it | kk) != 0 ? 1u : 0u);
                    } else {
                        const uint64_t da = dev::smem_desc_kmajor(st, ROW);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            dev::tc_mma_bf16<1>(d_tmem, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), idesc,
                                                (it | kk) != 0 ? 1u : 0u);
                    }
                    dev::tc_commit<1>(dev::smem_u32(&empty[stage]));
                    next_stage();
                }
                if (!ok) break;
                dev::tc_commit<1>(dev::smem_u32(&tfull[buf]));
            }
            // All tcgen05 operations issued by this thread must finish before TMEM is freed.
            dev::tc_commit<1>(dev::smem_u32(drain));
            if (!dev::mbar_wait_bounded(dev::smem_u32(drain), 0, nullptr, kCmTimeoutNs))
                cm_error(kErrTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp >= 4 && warp < 4 + kCmEpiWarps) {
        // ------------------------------------------------------------ epilogue
        // TMEM lane = output channel, column = pixel.  Warps w, w + 4 and w + 8 share
        // lane quarter w % 4 (32 channels) and take every third 16-pixel chunk in turn;
        // each thread owns one channel, transposed to NHWC through shared memory.
        const int ew = warp & 3;
        const int half = (warp - 4) >> 2;  // which of the quarter's warps: 0, 1 or 2
        uint8_t *my_stg = sm_stg + (warp - 4) * 2 * kCmStgBytes;
        const int ch_w0 = ct * 128 + ew * 32;  // warp's first channel
        const int ch = ch_w0 + lane;
        const float hs = ch < a.c_out ? 0.5f * __ldg(a.scale + ch) : 0.f;
        const float hb = ch < a.c_out ? 0.5f * __ldg(a.bias + ch) : 0.f;
        int sbuf = 0;
        CmIter<XMODE> iter(a, jcta);
        CmUnit u;
        for (int lt = 0; iter.get(a, u); ++lt) {
            const int buf = lt & 1;
            const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
            int okw = 1;
            if (lane == 0)
                okw = dev::mbar_wait_bounded(dev::smem_u32(&tfull[buf]), tparity, abort_flag, a.wait_ns) ? 1 : 0;
            okw = __shfl_sync(0xffffffffu, okw, 0);
            if (!okw) {
                if (lane == 0 && !*abort_flag) cm_error(kErrTimeoutEpilogue, abort_flag);
                break;
            }
            dev::tc_fence_after_sync();
            const int nchunks = (u.np + kCmChunk - 1) / kCmChunk;
            const uint32_t t_lane = tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(wcols + buf * a.unit_px);
            if (half >= nchunks || ch_w0 >= a.c_out) {
                // A unit of one chunk, or a lane quarter past the last output channel, leaves
                // this warp nothing to read or store.
                dev::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                continue;
            }
#pragma unroll 1
            for (int j = half; j < nchunks; j += kCmEpiWarps / 4) {
                uint32_t v[kCmChunk];
                dev::tmem_ld_32x32b_x16(t_lane + (uint32_t)(j * kCmChunk), v);
                dev::tmem_ld_wait();
                dev::reg_fence16(v);
                if (j + kCmEpiWarps / 4 >= nchunks) {
                    // This warp's last chunk is in registers: release the accumulator.
                    dev::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                }
                if (lane == 0) dev::bulk_wait_group_read<1>();  // the buffer's previous store has read it
                __syncwarp();
                // Staging rows: row pp holds pixel pp's 32 channels, one per lane.
                const uint32_t sb = dev::smem_u32(my_stg + sbuf * kCmStgBytes);
                auto activate = [&](auto mode_c) {
                    constexpr int md = decltype(mode_c)::value;
#pragma unroll
                    for (int pp = 0; pp < kCmChunk; ++pp)
                        dev::sts_u16(sb + (uint32_t)((pp * 32 + lane) * 2),
                                     __bfloat16_as_ushort(__float2bfloat16_rn(
                                         dev::epilogue_from_half(__uint_as_float(v[pp]), hs, hb, md))));
                };
                if constexpr (EPI == kEpiCmSilu) {
                    activate(std::integral_constant<int, kEpiSilu>{});
                } else {
                    switch (emode) {
                    case kEpiConvOnly: activate(std::integral_constant<int, kEpiConvOnly>{}); break;
                    case kEpiBn: activate(std::integral_constant<int, kEpiBn>{}); break;
                    case kEpiRelu: activate(std::integral_constant<int, kEpiRelu>{}); break;
                    default: activate(std::integral_constant<int, kEpiSilu>{}); break;
                    }
                }
                dev::fence_proxy_async_shared();
                __syncwarp();
                const int px0 = u.p0 + j * kCmChunk;
                if (lane == 0) {
                    dev::tma_store_2d(&tm_y, sb, ch_w0, px0);  // TMA clips channels >= c_out and pixels >= m
                    dev::bulk_commit_group();
                }
                sbuf ^= 1;
            }
        }
        if (lane == 0) dev::bulk_wait_group<0>();
        __syncwarp();
    }

    dev::tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        dev::tc_fence_after_sync();
        dev::tmem_dealloc<1>(tmem_base, 512);
    }
}

struct CmMaps {
    CUtensorMap x, w, y;
};

template <int BK, int EPI, bool WRES, int XMODE>
cudaError_t launch_cm(const ConvProblem &p, const TcPlan &plan, const CmMaps &maps, cudaStream_t stream)
{
    auto kern = tc_cmajor_kernel<BK, EPI, WRES, XMODE>;
    static std::mutex mu;
    static unsigned long long done = 0;  // bit per device ordinal (< 64)
    int device = 0;
    cudaError_t st = cudaGetDevice(&device);
    if (st != cudaSuccess) return st;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long bit = device < 64 ? (1ull << device) : 0ull;
        if (!(done & bit) || bit == 0) {
            st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCmSmemLimit);
            if (st != cudaSuccess) return st;
            done |= bit;
        }
    }
    CmArgs a;
    a.scale = p.scale;
    a.bias = p.bias;
    a.c = p.c;
    a.c_out = p.c_out;
    a.m = (int)p.m;
    a.ho = p.ho;
    a.wo = p.wo;
    a.howo = p.ho * p.wo;
    a.stride_h = p.stride_h;
    a.stride_w = p.stride_w;
    a.pad_h = p.pad_h;
    a.pad_w = p.pad_w;
    a.s = p.s;
    a.c_chunks = plan.c_chunks;
    a.k_iters = plan.k_iters;
    a.ctas_per_tile = plan.cm_ctas_per_tile;
    a.unit_px = plan.cm_unit_px;
    a.unit_rows = plan.cm_unit_rows;
    a.groups = plan.cm_unit_rows > 0 ? (p.ho + plan.cm_unit_rows - 1) / plan.cm_unit_rows : 0;
    a.stages = plan.stages;
    a.stage_bytes = plan.cm_stage_bytes;
    a.a_bytes = plan.cm_a_bytes;
    a.epi_mode = p.epi_mode;
    a.wait_ns = p.wait_timeout_ns > 0 ? (unsigned long long)p.wait_timeout_ns : kCmTimeoutNs;
    return launch_overlapped(kern, dim3((unsigned)plan.grid), dim3(kCmThreads), (size_t)plan.smem_bytes, stream, 1,
                             maps.x, maps.w, maps.y, a);
}

// Tensor maps of recent calls, keyed by pointers, shape, x mode and unit geometry.  The
// x mode is part of the key: an im2col load issued with a tiled map (or the reverse) is
// an illegal instruction, and two modes can share every other field (a 1x1 layer's
// matrix-row units and its im2col units may have the same pixel count).
struct CmKey {
    const void *x, *w, *y;
    int dims[11];
    int xmode, unit_px, unit_rows, block_k, device;
    bool operator==(const CmKey &o) const
    {
        if (x != o.x || w != o.w || y != o.y || xmode != o.xmode || unit_px != o.unit_px ||
            unit_rows != o.unit_rows || block_k != o.block_k || device != o.device)
            return false;
        for (int i = 0; i < 11; ++i)
            if (dims[i] != o.dims[i]) return false;
        return true;
    }
};

struct CmCache {
    static constexpr int kSlots = 32;
    std::mutex mu;
    CmKey keys[kSlots];
    CmMaps maps[kSlots];
    bool used[kSlots] = {};
    int next = 0;
};

CmCache g_cm_cache;

cudaError_t cm_maps(const ConvProblem &p, const TcPlan &plan, CmMaps *out)
{
    CmKey k{};
    k.x = p.x;
    k.w = p.w;
    k.y = p.y;
    const int d[11] = {p.n, p.h, p.w_in, p.c, p.c_out, p.r, p.s, p.stride_h, p.stride_w, p.pad_h, p.pad_w};
    for (int i = 0; i < 11; ++i) k.dims[i] = d[i];
    k.xmode = plan.cm_xmode;
    k.unit_px = plan.cm_unit_px;
    k.unit_rows = plan.cm_unit_rows;
    k.block_k = plan.block_k;
    cudaError_t st = cudaGetDevice(&k.device);
    if (st != cudaSuccess) return st;
    {
        std::lock_guard<std::mutex> lock(g_cm_cache.mu);
        for (int i = 0; i < CmCache::kSlots; ++i)
            if (g_cm_cache.used[i] && g_cm_cache.keys[i] == k) {
                *out = g_cm_cache.maps[i];
                return cudaSuccess;
            }
    }
    if (plan.cm_xmode == kXRows)
        st = tc_encode_x_rows(p, plan.block_k, plan.cm_unit_rows, &out->x);
    else if (plan.cm_xmode == kXMatrix)
        st = tc_encode_x_matrix(p, plan.block_k, plan.cm_unit_px, &out->x);
    else
        st = tc_encode_x_im2col(p, plan.block_k, plan.cm_unit_px, &out->x);
    if (st == cudaSuccess) st = tc_encode_w_tile(p, plan.block_k, 128, &out->w);
    if (st == cudaSuccess) st = tc_encode_y_rows(p, p.y, 32, kCmChunk, &out->y);
    if (st != cudaSuccess) return st;
    std::lock_guard<std::mutex> lock(g_cm_cache.mu);
    const int slot = g_cm_cache.next;
    g_cm_cache.next = (slot + 1) % CmCache::kSlots;
    g_cm_cache.keys[slot] = k;
    g_cm_cache.maps[slot] = *out;
    g_cm_cache.used[slot] = true;
    return cudaSuccess;
}

template <int EPI, bool WRES, int XMODE>
cudaError_t dispatch_bk(const ConvProblem &p, const TcPlan &plan, const CmMaps &maps, cudaStream_t stream)
{
    switch (plan.block_k) {
    case 64: return launch_cm<64, EPI, WRES, XMODE>(p, plan, maps, stream);
    case 32: return launch_cm<32, EPI, WRES, XMODE>(p, plan, maps, stream);
    case 16: return launch_cm<16, EPI, WRES, XMODE>(p, plan, maps, stream);
    default: return cudaErrorInvalidConfiguration;
    }
}

template <int EPI, bool WRES>
cudaError_t dispatch_x(const ConvProblem &p, const TcPlan &plan, const CmMaps &maps, cudaStream_t stream)
{
    switch (plan.cm_xmode) {
    case kXRows: return dispatch_bk<EPI, WRES, kXRows>(p, plan, maps, stream);
    case kXMatrix: return dispatch_bk<EPI, WRES, kXMatrix>(p, plan, maps, stream);
    default: return dispatch_bk<EPI, WRES, kXIm2col>(p, plan, maps, stream);
    }
}

template <int EPI>
cudaError_t dispatch_cm(const ConvProblem &p, const TcPlan &plan, const CmMaps &maps, cudaStream_t stream)
{
    return plan.cm_wres ? dispatch_x<EPI, true>(p, plan, maps, stream) : dispatch_x<EPI, false>(p, plan, maps, stream);
}

}  // namespace

bool cmajor_fill_plan(const ConvProblem &p, int sm_count, int wres, int xrows, TcPlan *t)
{
    // The bf16 output with the layer's own or a run-time activation; no residual.
    if (p.out_fp8 || p.residual != nullptr) return false;
    if (p.m > 0x7fffffffLL - 256) return false;
    const int block_k = p.c % 64 == 0 ? 64 : (p.c % 32 == 0 ? 32 : 16);
    const int c_chunks = (p.c + block_k - 1) / block_k;
    const int k_iters = p.r * p.s * c_chunks;
    const int wcols = wres ? k_iters * block_k / 2 : 0;
    // Two accumulators next to the resident weights, or two of at most 256 pixels.
    const int unit_max = std::min(256, (512 - wcols) / 2 / 16 * 16);
    if (unit_max < 64) return false;
    const int n_ctiles = (p.c_out + 127) / 128;
    if (n_ctiles > 4 || sm_count < n_ctiles) return false;
    const int per_tile = sm_count / n_ctiles;
    // A 1x1 layer at stride 1 without padding reads x as its [M][C] matrix ("row boxes"
    // then means tiled boxes of matrix rows, on pixel units).
    const bool matrix = p.r == 1 && p.s == 1 && p.stride_h == 1 && p.stride_w == 1 && p.pad_h == 0 && p.pad_w == 0;
    int xmode = kXIm2col, unit_px = 0, unit_rows = 0;
    if (xrows && !matrix) {
        // Row boxes: whole output rows of one image per unit; the view (stride*C, W/stride, H, N)
        // needs W divisible by the stride, equal strides (the H traversal stride is the conv's)
        // and at most 256 output columns.  Rows per unit: the count (units of a multiple of
        // 16 pixels, the short last group as well) that gives the busiest CTA the least work.
        if (p.stride_w != p.stride_h || p.stride_w > 8 || p.w_in % p.stride_w != 0) return false;
        if (p.wo > 256 || p.wo > unit_max || (long long)p.stride_h * (p.r - 1) + 1 > 256) return false;
        const long long images = p.m / ((long long)p.ho * p.wo);
        long long best = -1;
        for (int rows = std::min(unit_max / p.wo, p.ho); rows >= 1; --rows) {
            if ((rows * p.wo) % 16 != 0 || (p.ho % rows) * p.wo % 16 != 0) continue;
            // Each unit also costs a fixed pipeline fill and drain, taken as 64 pixels' worth.
            const long long units = images * ((p.ho + rows - 1) / rows);
            const long long cost = (units + per_tile - 1) / per_tile * (rows * p.wo + 64);
            if (best < 0 || cost < best) {
                best = cost;
                unit_rows = rows;
            }
        }
        if (unit_rows == 0) return false;
        xmode = kXRows;
        unit_px = unit_rows * p.wo;
    } else {
        // Pixel units: the largest share, in 16-pixel chunks, cut into equal units of at most unit_max.
        if (xrows && matrix) xmode = kXMatrix;
        const long long chunks = (p.m + kCmChunk - 1) / kCmChunk;
        const long long share = (chunks + per_tile - 1) / per_tile;
        const long long units = (share * kCmChunk + unit_max - 1) / unit_max;
        unit_px = (int)((share + units - 1) / units) * kCmChunk;
    }
    const int x_bytes = unit_px * block_k * 2;
    const int a_bytes = wres ? 0 : (128 * block_k * 2 + 1023) / 1024 * 1024;
    const int stage_bytes = wres ? (std::max(x_bytes, 128 * block_k * 2) + 1023) / 1024 * 1024
                                 : a_bytes + (x_bytes + 1023) / 1024 * 1024;
    const int fixed = 1024 + kCmEpiWarps * 2 * kCmStgBytes + 512;
    const int stages = std::min(kCmMaxStages, (kCmSmemLimit - fixed) / stage_bytes);
    if (stages < 3) return false;
    TcPlan out{};
    out.block_n = 128;  // channels per tile
    out.block_k = block_k;
    out.stages = stages;
    out.c_chunks = c_chunks;
    out.k_iters = k_iters;
    out.m_tiles = xmode == kXRows ? (int)(p.m / ((long long)p.ho * p.wo)) * ((p.ho + unit_rows - 1) / unit_rows)
                                  : (int)((p.m + unit_px - 1) / unit_px);
    out.n_tiles = n_ctiles;
    out.tiles = out.m_tiles * n_ctiles;
    out.grid = per_tile * n_ctiles;
    out.smem_bytes = fixed + stages * stage_bytes;
    out.swap_ab = 1;
    out.cmajor = 1;
    out.cm_wres = wres ? 1 : 0;
    out.cm_xmode = xmode;
    out.cm_unit_px = unit_px;
    out.cm_unit_rows = unit_rows;
    out.cm_ctas_per_tile = per_tile;
    out.cm_stage_bytes = stage_bytes;
    out.cm_a_bytes = a_bytes;
    *t = out;
    return true;
}

cudaError_t cmajor_launch(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream)
{
    CmMaps maps;
    cudaError_t st = cm_maps(p, plan, &maps);
    if (st != cudaSuccess) return st;
    if (p.epi_mode != kEpiSilu) return dispatch_cm<kEpiCmMode>(p, plan, maps, stream);
    return dispatch_cm<kEpiCmSilu>(p, plan, maps, stream);
}

cudaError_t cmajor_read_and_clear_error(cudaStream_t stream, unsigned int *out)
{
    unsigned int host = 0;
    cudaError_t st = cudaMemcpyFromSymbolAsync(&host, g_cmajor_error, sizeof host, 0, cudaMemcpyDeviceToHost, stream);
    if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    if (st != cudaSuccess) return st;
    if (host != 0) {
        const unsigned int zero = 0;
        st = cudaMemcpyToSymbolAsync(g_cmajor_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
        if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    }
    *out = host;
    return st;
}

}  // namespace cbs
