// fold.cu -- BatchNorm fold to one scale and one bias per output channel.
// ("Fusing an Epilogue", kernels book: batch norm reduces to a multiply and an
// add, loaded inside the fused kernel as one scale and one bias per channel.)
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

// Several layers' folds in one launch: 128 channels per block, the blocks of
// layer i starting at first_block[i].
__global__ void bn_fold_batch_kernel(const __grid_constant__ FoldBatch fb)
{
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();
    int layer = 0;
    while (layer + 1 < fb.count && (int)blockIdx.x >= fb.first_block[layer + 1]) ++layer;
    const FoldLayer &L = fb.layer[layer];
    const int k = ((int)blockIdx.x - fb.first_block[layer]) * blockDim.x + threadIdx.x;
    if (k >= L.c_out) return;
    const double sc = (double)L.gamma[k] / sqrt((double)L.var[k] + (double)L.eps);
    L.scale[k] = (float)sc;
    L.bias[k] = (float)((double)L.beta[k] - (double)L.mean[k] * sc);
}

}  // namespace

cudaError_t fold_batch_launch(const FoldLayer *layers, int count, cudaStream_t stream)
{
    const int threads = 128;
    for (int base = 0; base < count; base += kFoldBatchMax) {
        FoldBatch fb{};
        fb.count = count - base < kFoldBatchMax ? count - base : kFoldBatchMax;
        int blocks = 0;
        for (int i = 0; i < fb.count; ++i) {
            fb.layer[i] = layers[base + i];
            fb.first_block[i] = blocks;
            blocks += (fb.layer[i].c_out + threads - 1) / threads;
        }
        if (blocks == 0) continue;
        cudaError_t e = launch_overlapped(bn_fold_batch_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, 1,
                                          fb);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t fold_launch(const float *gamma, const float *beta, const float *mean, const float *var,
                        float eps, int c_out, float *scale, float *bias, cudaStream_t stream)
{
    const int threads = 128;
    return launch_overlapped(bn_fold_kernel, dim3((unsigned)((c_out + threads - 1) / threads)), dim3(threads), 0,
                             stream, 1, gamma, beta, mean, var, eps, c_out, scale, bias);
}

}  // namespace cbs
