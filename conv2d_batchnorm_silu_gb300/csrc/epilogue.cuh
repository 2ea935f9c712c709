// epilogue.cuh -- the fused epilogue arithmetic shared by every forward kernel:
// per-channel BatchNorm multiply/add, SiLU, and the narrowing cast to bf16.
// ("Fusing an Epilogue", kernels book, section "The shape of it":
//  acc = acc*bn_scale + bn_bias; acc = acc*sigmoid(acc); store acc.)
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace cbs {
namespace dev {

// z = acc*scale + bias;  SiLU(z) = z*sigmoid(z) = z / (1 + e^(-z)).
// __expf and __fdividef are the CUDA fast intrinsics (relative error around
// 2^-21); for z below about -88, e^(-z) overflows to +inf and the quotient is
// -0, the limit of SiLU.  The result is rounded to bf16 afterwards, which
// dominates the error (relative 2^-9).
__device__ __forceinline__ float bn_silu(float acc, float scale, float bias)
{
    const float z = fmaf(acc, scale, bias);
    return __fdividef(z, 1.0f + __expf(-z));
}

// Two floats -> packed bf16x2 (round to nearest even), `lo` in the low half,
// which is the lower address in memory.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace dev
}  // namespace cbs
