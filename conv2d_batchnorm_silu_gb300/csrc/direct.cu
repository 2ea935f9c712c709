// direct.cu -- fused conv2d + BatchNorm + SiLU on the CUDA cores, any shape.
//
// The "scalar" member of the family in "Fusing an Epilogue" (kernels book,
// section "Three kernels for one operation": one output element per lane, no
// set-up cost): here one thread owns one output pixel and a group of 16
// output channels, so the 16 accumulators stay in registers through the
// whole (r, s, c) reduction and the epilogue (BN multiply/add, SiLU, bf16
// cast) runs on them before the single store.  The block's 16 filters are
// staged in shared memory as fp32, [tap][16], in chunks, and every thread
// reads them as broadcast float4s.  It serves shapes the tensor-core kernel
// does not take (c % 16 != 0, e.g. a 3-channel stem; c_out % 8 != 0); common
// small filters use a fully unrolled variant (direct_small_kernel).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {
namespace {

constexpr int KB = kDirectBlockN;     // output channels per thread
constexpr int QCH = 512;              // filter taps (r, s, c) staged per chunk: 32 KB

struct DirectArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *w;
    const float *scale;
    const float *bias;
    __nv_bfloat16 *y;
    long long m;
    int h, w_in, c, c_out, r, s;
    int stride_h, stride_w, pad_h, pad_w, ho, wo;
    int epi_mode;   // EpiMode applied to the accumulator
    const __nv_bfloat16 *residual;  // nullable: bf16 [m][c_out] added after the activation
    int out_fp8;    // 1: y holds fp8 e4m3 bytes
};

// Epilogue on the registers: BN multiply/add, activation, optional residual,
// bf16, 16-byte stores when the channel run allows.
__device__ __forceinline__ void store_outputs(const DirectArgs &a, long long m, int k0, const float *acc)
{
    if (a.out_fp8) {
        unsigned char *y8 = reinterpret_cast<unsigned char *>(a.y) + m * a.c_out + k0;
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if (k0 + j < a.c_out)
                y8[j] = dev::to_e4m3(dev::epilogue_value(acc[j], __ldg(a.scale + k0 + j), __ldg(a.bias + k0 + j),
                                                         a.epi_mode));
        return;
    }
    __nv_bfloat16 *yp = a.y + m * a.c_out + k0;
    const __nv_bfloat16 *rp = a.residual != nullptr ? a.residual + m * a.c_out + k0 : nullptr;
    if (k0 + KB <= a.c_out && (a.c_out % 8) == 0) {
        float f[KB];
#pragma unroll
        for (int j = 0; j < KB; ++j)
            f[j] = dev::epilogue_value(acc[j], __ldg(a.scale + k0 + j), __ldg(a.bias + k0 + j), a.epi_mode);
        if (rp != nullptr) {
#pragma unroll
            for (int j = 0; j < KB; j += 8) dev::add_residual8(f + j, rp + j);
        }
        uint32_t packed[KB / 2];
#pragma unroll
        for (int j = 0; j < KB; j += 2) packed[j / 2] = dev::pack_bf16x2(f[j], f[j + 1]);
        uint4 *dst = reinterpret_cast<uint4 *>(yp);
#pragma unroll
        for (int v = 0; v < KB / 8; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
    } else {
#pragma unroll
        for (int j = 0; j < KB; ++j)
            if (k0 + j < a.c_out) {
                float f = dev::epilogue_value(acc[j], __ldg(a.scale + k0 + j), __ldg(a.bias + k0 + j), a.epi_mode);
                if (rp != nullptr) f += __bfloat162float(rp[j]);
                yp[j] = __float2bfloat16_rn(f);
            }
    }
}

__global__ void __launch_bounds__(kDirectThreads)
    direct_conv_bn_silu_kernel(const DirectArgs a)
{
    __shared__ __align__(16) float wsm[QCH][KB];
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    const long long m = (long long)blockIdx.x * kDirectThreads + threadIdx.x;
    const int k0 = blockIdx.y * KB;
    const bool active = m < a.m;
    int ow = 0, oh = 0, img = 0;
    if (active) {
        ow = (int)(m % a.wo);
        const long long t = m / a.wo;
        oh = (int)(t % a.ho);
        img = (int)(t / a.ho);
    }
    float acc[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) acc[j] = 0.f;

    const int taps = a.r * a.s * a.c;
    for (int q0 = 0; q0 < taps; q0 += QCH) {
        const int qn = min(QCH, taps - q0);
        __syncthreads();
        for (int i = threadIdx.x; i < qn * KB; i += kDirectThreads) {
            const int q = i / KB, j = i - q * KB;
            const int k = k0 + j;
            wsm[q][j] = k < a.c_out ? __bfloat162float(a.w[(long long)k * taps + q0 + q]) : 0.f;
        }
        __syncthreads();
        if (active) {
            int c = q0 % a.c;
            int rs = q0 / a.c;
            int s = rs % a.s;
            int r = rs / a.s;
            for (int q = 0; q < qn; ++q) {
                const int ih = oh * a.stride_h - a.pad_h + r;
                const int iw = ow * a.stride_w - a.pad_w + s;
                if (ih >= 0 && ih < a.h && iw >= 0 && iw < a.w_in) {
                    const float xv = __bfloat162float(
                        a.x[(((long long)img * a.h + ih) * a.w_in + iw) * a.c + c]);
                    const float4 *wq = reinterpret_cast<const float4 *>(wsm[q]);
#pragma unroll
                    for (int j4 = 0; j4 < KB / 4; ++j4) {
                        const float4 wv = wq[j4];
                        acc[4 * j4 + 0] = fmaf(xv, wv.x, acc[4 * j4 + 0]);
                        acc[4 * j4 + 1] = fmaf(xv, wv.y, acc[4 * j4 + 1]);
                        acc[4 * j4 + 2] = fmaf(xv, wv.z, acc[4 * j4 + 2]);
                        acc[4 * j4 + 3] = fmaf(xv, wv.w, acc[4 * j4 + 3]);
                    }
                }
                if (++c == a.c) {
                    c = 0;
                    if (++s == a.s) {
                        s = 0;
                        ++r;
                    }
                }
            }
        }
    }
    if (!active) return;
    store_outputs(a, m, k0, acc);
}

// Small filters with a compile-time shape (R x S taps of C channels): every
// thread issues all of its receptive-field loads before the first FMA, so a
// thread waits for memory once instead of once per tap (the generic kernel's
// tap loop is a chain of dependent load latencies).  C % 8 == 0 uses 16-byte
// vector loads.  Used for 3-channel stems and other thin-input layers.
template <int R, int S, int C, int NT>
__global__ void __launch_bounds__(NT) direct_small_kernel(const DirectArgs a)
{
    constexpr int TAPS = R * S * C;
    __shared__ __align__(16) float wsm[TAPS][KB];
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    const int k0 = blockIdx.y * KB;
    for (int i = threadIdx.x; i < TAPS * KB; i += NT) {
        const int q = i / KB, j = i - (i / KB) * KB;
        const int k = k0 + j;
        wsm[q][j] = k < a.c_out ? __bfloat162float(a.w[(long long)k * TAPS + q]) : 0.f;
    }
    const long long m = (long long)blockIdx.x * NT + threadIdx.x;
    const bool active = m < a.m;
    int ow = 0, oh = 0, img = 0;
    if (active) {
        ow = (int)(m % a.wo);
        const long long t = m / a.wo;
        oh = (int)(t % a.ho);
        img = (int)(t / a.ho);
    }
    // Gather the receptive field (zeros in the padding), all loads independent.
    constexpr int VEC = (C % 8 == 0) ? C / 8 : 0;  // 16-byte vectors per tap
    uint4 xv[VEC > 0 ? R * S * VEC : 1];
    unsigned short xs[VEC > 0 ? 1 : TAPS];
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int ih = oh * a.stride_h - a.pad_h + r;
            const int iw = ow * a.stride_w - a.pad_w + s;
            const bool in = active && ih >= 0 && ih < a.h && iw >= 0 && iw < a.w_in;
            const __nv_bfloat16 *px = a.x + (((long long)img * a.h + ih) * a.w_in + iw) * C;
            if constexpr (VEC > 0) {
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    xv[(r * S + s) * VEC + v] =
                        in ? __ldg(reinterpret_cast<const uint4 *>(px) + v) : make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
                for (int c = 0; c < C; ++c)
                    xs[(r * S + s) * C + c] = in ? __ldg(reinterpret_cast<const unsigned short *>(px) + c)
                                                 : (unsigned short)0;
            }
        }
    }
    __syncthreads();
    float acc[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) acc[j] = 0.f;
#pragma unroll
    for (int q = 0; q < TAPS; ++q) {
        float xf;
        if constexpr (VEC > 0) {
            const uint32_t *words = reinterpret_cast<const uint32_t *>(&xv[q / 8]);
            const uint32_t word = words[(q % 8) / 2];
            xf = __uint_as_float((q % 2) ? (word & 0xffff0000u) : (word << 16));
        } else {
            xf = __uint_as_float((uint32_t)xs[q] << 16);
        }
        const float4 *wq = reinterpret_cast<const float4 *>(wsm[q]);
#pragma unroll
        for (int j4 = 0; j4 < KB / 4; ++j4) {
            const float4 wv = wq[j4];
            acc[4 * j4 + 0] = fmaf(xf, wv.x, acc[4 * j4 + 0]);
            acc[4 * j4 + 1] = fmaf(xf, wv.y, acc[4 * j4 + 1]);
            acc[4 * j4 + 2] = fmaf(xf, wv.z, acc[4 * j4 + 2]);
            acc[4 * j4 + 3] = fmaf(xf, wv.w, acc[4 * j4 + 3]);
        }
    }
    if (!active) return;
    store_outputs(a, m, k0, acc);
}

constexpr int kSmallThreads = 64;

template <int R, int S, int C>
bool try_small(const ConvProblem &p, const DirectArgs &a, cudaStream_t stream, cudaError_t *err)
{
    if (p.r != R || p.s != S || p.c != C) return false;
    const long long bx = (p.m + kSmallThreads - 1) / kSmallThreads;
    if (bx > 0x7fffffffLL) return false;
    dim3 grid((unsigned)bx, (unsigned)((p.c_out + KB - 1) / KB));
    if (grid.y > 65535) return false;
    *err = launch_overlapped(direct_small_kernel<R, S, C, kSmallThreads>, grid, dim3(kSmallThreads), 0, stream,
                             1, a);
    return true;
}

}  // namespace

bool direct_small_available(int r, int s, int c)
{
    return r == 3 && s == 3 && (c == 1 || c == 3 || c == 4 || c == 8 || c == 16);
}

cudaError_t direct_launch(const ConvProblem &p, cudaStream_t stream)
{
    DirectArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(p.x);
    a.w = static_cast<const __nv_bfloat16 *>(p.w);
    a.scale = p.scale;
    a.bias = p.bias;
    a.y = static_cast<__nv_bfloat16 *>(p.y);
    a.m = p.m;
    a.h = p.h;
    a.w_in = p.w_in;
    a.c = p.c;
    a.c_out = p.c_out;
    a.r = p.r;
    a.s = p.s;
    a.stride_h = p.stride_h;
    a.stride_w = p.stride_w;
    a.pad_h = p.pad_h;
    a.pad_w = p.pad_w;
    a.ho = p.ho;
    a.wo = p.wo;
    a.epi_mode = p.epi_mode;
    a.residual = static_cast<const __nv_bfloat16 *>(p.residual);
    a.out_fp8 = p.out_fp8;
    cudaError_t err = cudaSuccess;
    if (try_small<3, 3, 1>(p, a, stream, &err) || try_small<3, 3, 3>(p, a, stream, &err) ||
        try_small<3, 3, 4>(p, a, stream, &err) || try_small<3, 3, 8>(p, a, stream, &err) ||
        try_small<3, 3, 16>(p, a, stream, &err))
        return err;
    const long long bx = (p.m + kDirectThreads - 1) / kDirectThreads;
    if (bx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    dim3 grid((unsigned)bx, (unsigned)((p.c_out + KB - 1) / KB));
    if (grid.y > 65535) return cudaErrorInvalidConfiguration;
    return launch_overlapped(direct_conv_bn_silu_kernel, grid, dim3(kDirectThreads), 0, stream, 1, a);
}

}  // namespace cbs
