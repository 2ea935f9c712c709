// fold.cu -- BatchNorm fold to one scale and one bias per output channel.
// ("Fusing an Epilogue", kernels book: batch norm is "a multiply and an add",
// loaded inside the fused kernel as one scale and one bias per channel.)
//   scale = gamma / sqrt(var + eps), bias = beta - mean * scale,
// evaluated in double precision and rounded once to float.
#include <cuda_runtime.h>

#include "cbs_internal.h"
#include "ptx.cuh"

namespace cbs {
namespace {

__global__ void bn_fold_kernel(const float *__restrict__ gamma, const float *__restrict__ beta,
                               const float *__restrict__ mean, const float *__restrict__ var, float eps,
                               int c_out, float *__restrict__ scale, float *__restrict__ bias)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= c_out) return;
    const double sc = (double)gamma[k] / sqrt((double)var[k] + (double)eps);
    scale[k] = (float)sc;
    bias[k] = (float)((double)beta[k] - (double)mean[k] * sc);
}

}  // namespace

cudaError_t fold_launch(const float *gamma, const float *beta, const float *mean, const float *var,
                        float eps, int c_out, float *scale, float *bias, cudaStream_t stream)
{
    const int threads = 128;
    return launch_overlapped(bn_fold_kernel, dim3((unsigned)((c_out + threads - 1) / threads)), dim3(threads), 0,
                             stream, 1, gamma, beta, mean, var, eps, c_out, scale, bias);
}

}  // namespace cbs
