// tc_gather.cu -- fused conv2d + BatchNorm + SiLU on the tcgen05 tensor cores
// for thin inputs (C*R*S <= 64, e.g. a 3-channel stem), whose pixel rows are
// too narrow for TMA (a 6-byte pixel stride breaks its 16-byte stride rule).
//
// Same GEMM view as tc_conv.cu (M = output pixels, N = output channels,
// K = R*S*C ordered (r, s, c)), but the whole K fits one shared-memory row of
// KPAD = 32 or 64 bf16 (zero beyond R*S*C), so each output tile is one or two
// MMAs.  Per CTA:
//   warps 4..7  producers: one thread per output pixel of the 128-pixel tile
//               gathers its R*S*C receptive-field values straight from global
//               memory (zeros in the padding), packs them into its 64/128-byte
//               row of the swizzled A stage and arrives on the stage barrier
//               (after a proxy fence, so the tensor core sees the writes);
//   warp 8      MMA issuer: tcgen05.mma (M=128, N, K=16) against the weight tile
//               B, which stays in shared memory for the whole kernel;
//   warps 0..3  epilogue: tcgen05.ld of the accumulator, BN multiply/add, SiLU,
//               bf16, and one contiguous 2*N-byte store per pixel (consecutive
//               pixels are consecutive rows of y, so each warp stores 32 rows
//               back to back).
// The arithmetic per pixel is a handful of loads and stores: the layer stays
// bound by HBM traffic (x read once, y written once) rather than by the
// R*S*C*N fused multiply-adds a CUDA-core kernel would issue.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {

__device__ unsigned int g_gather_error = 0;

namespace {

constexpr uint64_t kGatherTimeoutNs = 2000000000ull;
constexpr int kGatherThreads = 288;  // 4 epilogue + 4 producer warps + the MMA warp
constexpr int kGatherStages = 4;

struct GatherArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *w;
    const float *scale;
    const float *bias;
    __nv_bfloat16 *y;
    int m, tiles;
    int h, w_in, c_out, ho, wo, howo;
    int stride_h, stride_w, pad_h, pad_w;
    int epi_mode;   // EpiMode applied to the accumulator
    const __nv_bfloat16 *residual;  // nullable: bf16 [m][c_out] added after the activation
};

template <int R, int S, int C, int N>
struct GatherCfg {
    static constexpr int TAPS = R * S * C;
    static constexpr int KPAD = TAPS <= 32 ? 32 : 64;
    static constexpr int ROW = KPAD * 2;                  // bytes per operand row = swizzle span
    static constexpr int A_BYTES = 128 * ROW;
    static constexpr int B_BYTES = ((N * ROW + 1023) / 1024) * 1024;
    static constexpr int TMEM_COLS = 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128);  // power of two
    static constexpr int SMEM = 1024 + kGatherStages * A_BYTES + B_BYTES + 256;
    static_assert(TAPS <= 64, "the receptive field must fit one 128-byte row");
    static_assert(N % 16 == 0 && N >= 16 && N <= 64, "UMMA N for M=128, epilogue width");
};

template <int ROW>
__device__ __forceinline__ uint32_t swz(uint32_t off)
{
    constexpr uint32_t mask = ROW == 128 ? 7u : (ROW == 64 ? 3u : 1u);
    return off ^ (((off >> 7) & mask) << 4);
}

__device__ __forceinline__ void gather_error(unsigned int bit, volatile int *abort_flag)
{
    atomicOr(&g_gather_error, bit);
    *abort_flag = 1;
}

template <int R, int S, int C, int N>
__global__ void __launch_bounds__(kGatherThreads, 2) tc_gather_conv_bn_silu_kernel(const GatherArgs a)
{
    using G = GatherCfg<R, S, C, N>;
    constexpr int KPAD = G::KPAD;
    constexpr int ROW = G::ROW;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + kGatherStages * G::A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_b + G::B_BYTES);
    uint64_t *full = bars;
    uint64_t *empty = full + kGatherStages;
    uint64_t *tfull = empty + kGatherStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kGatherStages; ++i) {
            dev::mbar_init(dev::smem_u32(&full[i]), 4);  // one arrival per producer warp
            dev::mbar_init(dev::smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&tfull[i]), 1);
            dev::mbar_init(dev::smem_u32(&tempty[i]), 4);
        }
        dev::mbar_init(dev::smem_u32(drain), 1);
        *abort_flag = 0;
        dev::fence_mbarrier_init();
    }
    if (warp == 8) {
        dev::tmem_alloc(dev::smem_u32(tmem_slot), G::TMEM_COLS);
        dev::tmem_relinquish_alloc_permit();
    }
    dev::tc_fence_before_sync();
    __syncthreads();
    dev::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();

    // Weight tile B: row k = output channel, K = (r, s, c) zero-padded to KPAD,
    // in the swizzled K-major layout the MMA descriptor describes.
    for (int i = threadIdx.x; i < N * (KPAD / 2); i += kGatherThreads) {
        const int k = i / (KPAD / 2), q2 = (i - k * (KPAD / 2)) * 2;
        uint32_t lo = 0, hi = 0;
        if (k < a.c_out) {
            const unsigned short *wp = reinterpret_cast<const unsigned short *>(a.w) + (size_t)k * G::TAPS;
            if (q2 < G::TAPS) lo = wp[q2];
            if (q2 + 1 < G::TAPS) hi = wp[q2 + 1];
        }
        *reinterpret_cast<uint32_t *>(sm_b + swz<ROW>((uint32_t)(k * ROW + q2 * 2))) = lo | (hi << 16);
    }
    dev::fence_proxy_async_shared();
    __syncthreads();

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ producers
        const int row = (warp - 4) * 32 + lane;  // pixel of the tile this thread gathers
        // Receptive field of this thread's pixel in tile t: all loads issued at
        // once (zeros in the padding).
        auto gather = [&](int t, unsigned short (&v)[G::TAPS]) {
            const int m = t * 128 + row;
            int img = 0, oh = 0, ow = 0;
            const bool active = t < a.tiles && m < a.m;
            if (active) {
                img = m / a.howo;
                const int rem = m - img * a.howo;
                oh = rem / a.wo;
                ow = rem - oh * a.wo;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    const int ih = oh * a.stride_h - a.pad_h + r;
                    const int iw = ow * a.stride_w - a.pad_w + s;
                    const bool in = active && ih >= 0 && ih < a.h && iw >= 0 && iw < a.w_in;
                    const unsigned short *px = reinterpret_cast<const unsigned short *>(a.x) +
                                               (((size_t)img * a.h + ih) * a.w_in + iw) * C;
#pragma unroll
                    for (int c = 0; c < C; ++c) v[(r * S + s) * C + c] = in ? __ldg(px + c) : (unsigned short)0;
                }
            }
        };
        int stage = 0;
        uint32_t phase = 0;
        unsigned short cur[G::TAPS], nxt[G::TAPS];
        gather(blockIdx.x, cur);
        for (int t = blockIdx.x; t < a.tiles && !*abort_flag; t += gridDim.x) {
            // Software pipeline: the next tile's loads are in flight while this
            // tile is packed into shared memory.
            gather(t + gridDim.x, nxt);
            int ok = 1;
            if (lane == 0)
                ok = dev::mbar_wait_bounded(dev::smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                            kGatherTimeoutNs)
                         ? 1
                         : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) gather_error(kErrTimeoutProducer, abort_flag);
                break;
            }
            uint8_t *arow = sm_a + stage * G::A_BYTES;
#pragma unroll
            for (int j = 0; j < ROW / 16; ++j) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int q = j * 8 + e * 2;
                    const uint32_t lo = q < G::TAPS ? cur[q < G::TAPS ? q : 0] : 0u;
                    const uint32_t hi = q + 1 < G::TAPS ? cur[q + 1 < G::TAPS ? q + 1 : 0] : 0u;
                    wv[e] = lo | (hi << 16);
                }
                *reinterpret_cast<uint4 *>(arow + swz<ROW>((uint32_t)(row * ROW + j * 16))) =
                    make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
            dev::fence_proxy_async_shared();  // generic-proxy writes -> tensor-core reads
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&full[stage]));
            if (++stage == kGatherStages) {
                stage = 0;
                phase ^= 1u;
            }
#pragma unroll
            for (int q = 0; q < G::TAPS; ++q) cur[q] = nxt[q];
        }
    } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = dev::idesc_bf16_f32(128, N);
            const uint64_t desc_a0 = dev::smem_desc_kmajor(dev::smem_u32(sm_a), ROW);
            const uint64_t desc_b = dev::smem_desc_kmajor(dev::smem_u32(sm_b), ROW);
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++lt) {
                const int buf = lt & 1;
                const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
                if (!dev::mbar_wait_bounded(dev::smem_u32(&tempty[buf]), tparity ^ 1u, abort_flag,
                                            kGatherTimeoutNs)) {
                    if (!*abort_flag) gather_error(kErrTimeoutMma, abort_flag);
                    break;
                }
                if (!dev::mbar_wait_bounded(dev::smem_u32(&full[stage]), phase, abort_flag, kGatherTimeoutNs)) {
                    if (!*abort_flag) gather_error(kErrTimeoutMma, abort_flag);
                    break;
                }
                dev::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * N);
                const uint64_t da = desc_a0 + (uint64_t)(stage * (G::A_BYTES >> 4));
#pragma unroll
                for (int kk = 0; kk < KPAD / 16; ++kk)
                    dev::tc_mma_bf16(d_tmem, da + (uint64_t)(2 * kk), desc_b + (uint64_t)(2 * kk), idesc,
                                     kk ? 1u : 0u);
                dev::tc_commit(dev::smem_u32(&empty[stage]));
                dev::tc_commit(dev::smem_u32(&tfull[buf]));
                if (++stage == kGatherStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            dev::tc_commit(dev::smem_u32(drain));
            if (!dev::mbar_wait_bounded(dev::smem_u32(drain), 0, nullptr, kGatherTimeoutNs))
                gather_error(kErrTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        // This thread's output channels never change: for narrow tiles keep scale/2
        // and bias/2 in registers, for wider ones read them (L1-resident) per use.
        constexpr int NREG = N <= 16 ? N : 1;
        float hs[NREG], hb[NREG];
#pragma unroll
        for (int j = 0; j < NREG; ++j) {
            hs[j] = j < a.c_out ? 0.5f * __ldg(a.scale + j) : 0.f;
            hb[j] = j < a.c_out ? 0.5f * __ldg(a.bias + j) : 0.f;
        }
        auto half_scale = [&](int j) {
            if constexpr (N <= 16) return hs[j];
            else return j < a.c_out ? 0.5f * __ldg(a.scale + j) : 0.f;
        };
        auto half_bias = [&](int j) {
            if constexpr (N <= 16) return hb[j];
            else return j < a.c_out ? 0.5f * __ldg(a.bias + j) : 0.f;
        };
        int lt = 0;
        for (int t = blockIdx.x; t < a.tiles; t += gridDim.x, ++lt) {
            const int buf = lt & 1;
            const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
            int ok = 1;
            if (lane == 0)
                ok = dev::mbar_wait_bounded(dev::smem_u32(&tfull[buf]), tparity, abort_flag, kGatherTimeoutNs) ? 1
                                                                                                               : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) gather_error(kErrTimeoutEpilogue, abort_flag);
                break;
            }
            dev::tc_fence_after_sync();
            uint32_t v[N];
            const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * N);
#pragma unroll
            for (int q = 0; q < N / 16; ++q) dev::tmem_ld_32x32b_x16(taddr + (uint32_t)(q * 16), v + q * 16);
            dev::tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < N / 16; ++q) dev::reg_fence16(v + q * 16);
            dev::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
            const int m = t * 128 + warp * 32 + lane;
            if (m < a.m) {
                uint32_t packed[N / 2];
                if (a.residual != nullptr) {
                    const __nv_bfloat16 *rp = a.residual + (size_t)m * a.c_out;
#pragma unroll
                    for (int j = 0; j < N; j += 2) {
                        const float r0 = j < a.c_out ? __bfloat162float(rp[j]) : 0.f;
                        const float r1 = j + 1 < a.c_out ? __bfloat162float(rp[j + 1]) : 0.f;
                        packed[j / 2] = dev::pack_bf16x2(
                            dev::epilogue_from_half(__uint_as_float(v[j]), half_scale(j), half_bias(j), a.epi_mode) + r0,
                            dev::epilogue_from_half(__uint_as_float(v[j + 1]), half_scale(j + 1), half_bias(j + 1),
                                                    a.epi_mode) + r1);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < N; j += 2)
                        packed[j / 2] = dev::pack_bf16x2(
                            dev::epilogue_from_half(__uint_as_float(v[j]), half_scale(j), half_bias(j), a.epi_mode),
                            dev::epilogue_from_half(__uint_as_float(v[j + 1]), half_scale(j + 1), half_bias(j + 1),
                                                    a.epi_mode));
                }
                __nv_bfloat16 *yp = a.y + (size_t)m * a.c_out;
                if (a.c_out == N) {
                    uint4 *dst = reinterpret_cast<uint4 *>(yp);
#pragma unroll
                    for (int q = 0; q < N / 8; ++q)
                        dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                } else {
                    const unsigned short *h16 = reinterpret_cast<const unsigned short *>(packed);
                    unsigned short *d16 = reinterpret_cast<unsigned short *>(yp);
                    for (int j = 0; j < a.c_out; ++j) d16[j] = h16[j];
                }
            }
        }
    }

    dev::tc_fence_before_sync();
    __syncthreads();
    if (warp == 8) {
        dev::tc_fence_after_sync();
        dev::tmem_dealloc(tmem_base, G::TMEM_COLS);
    }
}

template <int R, int S, int C, int N>
bool try_gather(const ConvProblem &p, int sm_count, cudaStream_t stream, cudaError_t *err)
{
    if (p.r != R || p.s != S || p.c != C || p.c_out > N || (N > 16 && p.c_out <= N - 16)) return false;
    using G = GatherCfg<R, S, C, N>;
    auto kern = tc_gather_conv_bn_silu_kernel<R, S, C, N>;
    static std::mutex mu;
    static unsigned long long done = 0;
    int device = 0;
    *err = cudaGetDevice(&device);
    if (*err != cudaSuccess) return true;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long bit = device < 64 ? (1ull << device) : 0ull;
        if (!(done & bit) || bit == 0) {
            *err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (*err != cudaSuccess) return true;
            done |= bit;
        }
    }
    GatherArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(p.x);
    a.w = static_cast<const __nv_bfloat16 *>(p.w);
    a.scale = p.scale;
    a.bias = p.bias;
    a.y = static_cast<__nv_bfloat16 *>(p.y);
    a.m = (int)p.m;
    a.tiles = (int)((p.m + 127) / 128);
    a.h = p.h;
    a.w_in = p.w_in;
    a.c_out = p.c_out;
    a.ho = p.ho;
    a.wo = p.wo;
    a.howo = p.ho * p.wo;
    a.stride_h = p.stride_h;
    a.stride_w = p.stride_w;
    a.pad_h = p.pad_h;
    a.pad_w = p.pad_w;
    a.epi_mode = p.epi_mode;
    a.residual = static_cast<const __nv_bfloat16 *>(p.residual);
    const int grid = a.tiles < 2 * sm_count ? a.tiles : 2 * sm_count;
    *err = launch_overlapped(kern, dim3((unsigned)grid), dim3(kGatherThreads), (size_t)G::SMEM, stream, 1, a);
    return true;
}

}  // namespace

bool gather_supported(const ConvProblem &p)
{
    if (p.m > 0x7fffffffLL - 128) return false;
    if (p.out_fp8) return false;  // the bf16 output only (the direct kernel writes fp8)
    const bool shape = p.r == 3 && p.s == 3 && (p.c == 1 || p.c == 3 || p.c == 4);
    return shape && p.c_out >= 1 && p.c_out <= 64;
}

cudaError_t gather_launch(const ConvProblem &p, int sm_count, cudaStream_t stream)
{
    cudaError_t err = cudaErrorInvalidConfiguration;
#define CBS_GATHER(C_)                                                                  \
    if (try_gather<3, 3, C_, 16>(p, sm_count, stream, &err) ||                          \
        try_gather<3, 3, C_, 32>(p, sm_count, stream, &err) ||                          \
        try_gather<3, 3, C_, 48>(p, sm_count, stream, &err) ||                          \
        try_gather<3, 3, C_, 64>(p, sm_count, stream, &err))                            \
        return err;
    CBS_GATHER(1) CBS_GATHER(3) CBS_GATHER(4)
#undef CBS_GATHER
    return err;
}

cudaError_t gather_read_and_clear_error(cudaStream_t stream, unsigned int *out)
{
    unsigned int host = 0;
    cudaError_t st = cudaMemcpyFromSymbolAsync(&host, g_gather_error, sizeof host, 0,
                                               cudaMemcpyDeviceToHost, stream);
    if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    if (st != cudaSuccess) return st;
    if (host != 0) {
        const unsigned int zero = 0;
        st = cudaMemcpyToSymbolAsync(g_gather_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
        if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    }
    *out = host;
    return st;
}

}  // namespace cbs
