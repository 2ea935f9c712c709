// unfused.cu -- the unfused comparator's elementwise steps.
//
// The fusion page contrasts one fused kernel with the sequence it replaces:
// the convolution writes its output to memory, a BatchNorm kernel reads it
// back and writes it again, and a SiLU kernel does the same once more
// ("Fusing an Epilogue", kernels book, sections "The problem" and "When not
// to fuse").  The convolution step is the forward kernel in conv-only mode;
// these two kernels are the other two steps:
//   t2[i] = bf16(t1[i] * scale[k] + bias[k]),  k = i mod c_out   (NHWC)
//   y[i]  = bf16(SiLU(t2[i]))
// Both are HBM-bound streams: 16-byte vector loads (evict-first: each input is
// read once) and plain stores (the next step may still find them in L2), one
// vector per thread (grid-stride beyond 2^22 blocks), with the per-channel
// scale/bias read as float4s when the channel count keeps a vector inside one
// pixel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// One 16-byte vector (8 channels of one pixel) per thread; c_out % 8 == 0.
__global__ void __launch_bounds__(kThreads) bn_apply_vec_kernel(const uint4 *__restrict__ t1,
                                                                const float *__restrict__ scale,
                                                                const float *__restrict__ bias,
                                                                uint4 *__restrict__ t2, long long vecs,
                                                                int c_out)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < vecs;
         i += (long long)gridDim.x * kThreads) {
        const int k0 = (int)((i * 8) % c_out);
        const float4 s0 = __ldg(reinterpret_cast<const float4 *>(scale + k0));
        const float4 s1 = __ldg(reinterpret_cast<const float4 *>(scale + k0 + 4));
        const float4 b0 = __ldg(reinterpret_cast<const float4 *>(bias + k0));
        const float4 b1 = __ldg(reinterpret_cast<const float4 *>(bias + k0 + 4));
        const uint4 v = __ldcs(t1 + i);
        uint4 o;
        o.x = dev::pack_bf16x2(fmaf(bf16_lo(v.x), s0.x, b0.x), fmaf(bf16_hi(v.x), s0.y, b0.y));
        o.y = dev::pack_bf16x2(fmaf(bf16_lo(v.y), s0.z, b0.z), fmaf(bf16_hi(v.y), s0.w, b0.w));
        o.z = dev::pack_bf16x2(fmaf(bf16_lo(v.z), s1.x, b1.x), fmaf(bf16_hi(v.z), s1.y, b1.y));
        o.w = dev::pack_bf16x2(fmaf(bf16_lo(v.w), s1.z, b1.z), fmaf(bf16_hi(v.w), s1.w, b1.w));
        t2[i] = o;
    }
}

// Any channel count: one element per thread.
__global__ void __launch_bounds__(kThreads) bn_apply_scalar_kernel(const __nv_bfloat16 *__restrict__ t1,
                                                                   const float *__restrict__ scale,
                                                                   const float *__restrict__ bias,
                                                                   __nv_bfloat16 *__restrict__ t2,
                                                                   long long count, int c_out)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < count;
         i += (long long)gridDim.x * kThreads) {
        const int k = (int)(i % c_out);
        t2[i] = __float2bfloat16_rn(fmaf(__bfloat162float(t1[i]), __ldg(scale + k), __ldg(bias + k)));
    }
}

__device__ __forceinline__ float silu_of(float z) { return dev::silu_from_half(0.5f * z); }

__global__ void __launch_bounds__(kThreads) silu_apply_vec_kernel(const uint4 *__restrict__ t2,
                                                                  uint4 *__restrict__ y, long long vecs)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < vecs;
         i += (long long)gridDim.x * kThreads) {
        const uint4 v = __ldcs(t2 + i);
        uint4 o;
        o.x = dev::pack_bf16x2(silu_of(bf16_lo(v.x)), silu_of(bf16_hi(v.x)));
        o.y = dev::pack_bf16x2(silu_of(bf16_lo(v.y)), silu_of(bf16_hi(v.y)));
        o.z = dev::pack_bf16x2(silu_of(bf16_lo(v.z)), silu_of(bf16_hi(v.z)));
        o.w = dev::pack_bf16x2(silu_of(bf16_lo(v.w)), silu_of(bf16_hi(v.w)));
        y[i] = o;
    }
}

__global__ void __launch_bounds__(kThreads) silu_apply_scalar_kernel(const __nv_bfloat16 *__restrict__ t2,
                                                                     __nv_bfloat16 *__restrict__ y,
                                                                     long long count)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    for (long long i = (long long)blockIdx.x * kThreads + threadIdx.x; i < count;
         i += (long long)gridDim.x * kThreads)
        y[i] = __float2bfloat16_rn(silu_of(__bfloat162float(t2[i])));
}

// One item per thread up to 2^22 blocks; beyond that each thread strides over several.
dim3 blocks_for(long long items)
{
    const long long b = (items + kThreads - 1) / kThreads;
    return dim3((unsigned)(b < (1LL << 22) ? b : (1LL << 22)));
}

}  // namespace

cudaError_t bn_apply_launch(const void *t1, const float *scale, const float *bias, void *t2, long long count,
                            int c_out, cudaStream_t stream)
{
    if (count <= 0) return cudaSuccess;
    if (c_out % 8 == 0)
        return launch_overlapped(bn_apply_vec_kernel, blocks_for(count / 8), dim3(kThreads), 0, stream, 1,
                                 static_cast<const uint4 *>(t1), scale, bias, static_cast<uint4 *>(t2),
                                 count / 8, c_out);
    return launch_overlapped(bn_apply_scalar_kernel, blocks_for(count), dim3(kThreads), 0, stream, 1,
                             static_cast<const __nv_bfloat16 *>(t1), scale, bias,
                             static_cast<__nv_bfloat16 *>(t2), count, c_out);
}

cudaError_t silu_apply_launch(const void *t2, void *y, long long count, cudaStream_t stream)
{
    if (count <= 0) return cudaSuccess;
    if (count % 8 == 0)
        return launch_overlapped(silu_apply_vec_kernel, blocks_for(count / 8), dim3(kThreads), 0, stream, 1,
                                 static_cast<const uint4 *>(t2), static_cast<uint4 *>(y), count / 8);
    return launch_overlapped(silu_apply_scalar_kernel, blocks_for(count), dim3(kThreads), 0, stream, 1,
                             static_cast<const __nv_bfloat16 *>(t2), static_cast<__nv_bfloat16 *>(y), count);
}

}  // namespace cbs
