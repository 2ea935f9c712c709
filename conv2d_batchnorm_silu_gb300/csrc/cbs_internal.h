// cbs_internal.h -- host-side types shared by the C ABI (capi.cu) and the kernel
// translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cbs {

// What the epilogue applies to the accumulator (a kernel argument, uniform
// over the launch).
enum EpiMode : int {
    kEpiSilu = 0,      // SiLU(acc*scale + bias): the fused layer
    kEpiConvOnly = 1,  // acc: the unfused comparator's first step stores t1 = conv(x, W)
    kEpiBn = 2,        // acc*scale + bias: BN (or a plain per-channel bias) without activation
    kEpiRelu = 3,      // max(acc*scale + bias, 0)
};

// One convolution call, with the derived GEMM view M = n*ho*wo, N = c_out, K = c*r*s.
struct ConvProblem {
    const void *x;
    const void *w;
    const float *scale;
    const float *bias;
    void *y;
    int n, h, w_in, c, c_out, r, s;
    int stride_h, stride_w, pad_h, pad_w;
    int ho, wo;
    long long m;    // output pixels
    int epi_mode;          // EpiMode: SiLU (the layer), conv only, BN only, BN + ReLU
    const void *residual;  // nullable bf16 NHWC [m][c_out], added after the activation
    long long wait_timeout_ns;  // > 0: bound on the tcgen05 kernel's pipeline waits (0: the 2 s default)
    int out_fp8;                // 1: y is fp8 e4m3 (one byte per element, round to nearest even, saturating)
};

// Tile configuration of the tcgen05 implicit GEMM.
struct TcPlan {
    int block_n;   // 16, 32, 64, 128 or 256 (UMMA N)
    int block_k;   // 16, 32 or 64 channels per stage (= swizzle width / 2 bytes)
    int stages;
    int c_chunks;  // ceil(c / block_k)
    int k_iters;   // r * s * c_chunks
    int m_tiles, n_tiles, tiles;
    int grid;
    int smem_bytes;
    int swap_ab;                  // 1: tile = 128 channels x block_n pixels, D = W * X^T
    int pair;                     // 1: clusters of two CTAs run the 2-CTA MMA, each holding half the weight tile
    int stream_k;                 // 1: K steps split evenly over the grid (see tc_conv.cu)
    int balanced;                 // swap_ab only: each CTA takes an equal run of 32-pixel chunks (see tc_conv.cu)
    long long workspace_bytes;    // stream-K partial tiles + flags (0 when not split)
    long long flag_bytes;         // the leading part of the workspace that must start zeroed
    // The channel-major kernel of tc_cmajor.cu (cmajor = 1): units of cm_unit_px pixels,
    // x in boxes of cm_unit_rows whole output rows (0: im2col boxes), the weight tile
    // resident in tensor memory (cm_wres = 1) or loaded with every K step.
    int cmajor;
    int cm_wres;
    int cm_xmode;                 // 0 im2col boxes, 1 row boxes, 2 boxes of the [M][C] matrix (1x1, stride 1)
    int cm_unit_px;
    int cm_unit_rows;
    int cm_ctas_per_tile;         // CTAs per 128-channel tile (the grid is this x channel tiles)
    int cm_stage_bytes;           // one pipeline stage
    int cm_a_bytes;               // streamed weights: the weight part of a stage
};

constexpr int kTcBlockM = 128;
// Epilogue warps per TMEM lane quarter of tc_conv.cu's kernel: three on 256-wide 2-CTA pair
// tiles (the last tile's epilogue runs with no K loop under it, and more warps hide its
// latency), two from 64 channels, one below.  The CTA has four other warps.
__host__ __device__ constexpr int tc_epi_warps_per_quarter(int block_n, bool pair)
{
    return (pair && block_n == 256) ? 3 : (block_n >= 64 ? 2 : 1);
}
__host__ __device__ constexpr int tc_threads(int block_n, bool pair)
{
    return 128 + 32 * 4 * tc_epi_warps_per_quarter(block_n, pair);
}
// Channel-major kernel of tc_cmajor.cu: producer, MMA, weight producer, one idle warp and
// twelve epilogue warps (three per TMEM lane quarter: the epilogue, not the loads, paced
// its units with eight).
constexpr int kCmEpiWarps = 12;
constexpr int kCmThreads = 128 + 32 * kCmEpiWarps;
// Stream-K slot words: a ready flag per (TMEM lane quarter, 32-column chunk) of a tile of up
// to 256 columns.
constexpr int kTcFlagsPerSlot = 32;

// Epilogue geometry of the tensor-core kernel for an N tile of `block_n`
// channels: `split` warps share each 32-row TMEM lane quarter (each takes
// block_n/split columns), processed `ec` columns at a time.
inline void tc_epilogue_geometry(int block_n, int *split, int *ec)
{
    *split = block_n >= 64 ? 2 : 1;
    const int cols = block_n / *split;
    *ec = cols < 32 ? cols : 32;
}
constexpr int kDirectThreads = 128;
constexpr int kDirectBlockN = 16;

// Launches `kern` on `stream` with programmatic stream serialization (the
// kernel may start while its predecessor drains; see grid_dependency_wait in
// ptx.cuh) and, when cluster_x > 1, clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, int cluster_x, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    cudaError_t st = cudaLaunchKernelEx(&cfg, kern, args...);
    if (st != cudaSuccess) return st;
    return cudaGetLastError();
}

// Planning (host only, no GPU needed).
bool tc_supported(const ConvProblem &p);
TcPlan tc_make_plan(const ConvProblem &p, int sm_count);
// Overrides of the planner's tcgen05 choices: -1 (block_n: 0) leaves a choice to the planner.
struct PlanRequest {
    int swap_ab, stream_k, pair, block_n;
    int balanced;  // channel-major tiles: -1 planner, 0 whole 256-pixel tiles, 1 equal runs of 32-pixel chunks
    int wres;      // -1 planner, 0 weights streamed with every tile, 1 weights resident in tensor memory
    int row_boxes; // -1 planner, 0 im2col boxes, 1 boxes of whole output rows (channel-major kernel)
};
// As tc_make_plan with the overrides in `rq` (nullable); -1 when the kernel cannot run
// them on this shape (e.g. stream-K shares shorter than one tile).
int tc_make_plan_request(const ConvProblem &p, int sm_count, const PlanRequest *rq, TcPlan *out);
// The channel-major kernel's plan (tc_cmajor.cu) with the weights resident in tensor memory
// or not and x in row boxes or im2col boxes; false when it cannot run that combination.
bool cmajor_fill_plan(const ConvProblem &p, int sm_count, int wres, int xrows, TcPlan *t);
cudaError_t cmajor_launch(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream);
cudaError_t cmajor_read_and_clear_error(cudaStream_t stream, unsigned int *out);
// Tensor maps shared by the tensor-core kernels (tc_conv.cu): x in im2col mode with boxes
// of `box_pixels` output pixels x block_k channels; a weight load of block_k channels of
// one filter tap for `rows` output channels; a tensor shaped like y, unswizzled boxes.
cudaError_t tc_encode_x_im2col(const ConvProblem &p, int block_k, int box_pixels, CUtensorMap *out);
// x viewed as (stride*C, W/stride, H, N) with boxes of block_k channels x wo view pixels x
// `rows` input rows taken every stride-th row (W divisible by the stride).
cudaError_t tc_encode_x_rows(const ConvProblem &p, int block_k, int rows, CUtensorMap *out);
// x of a 1x1 stride-1 layer as the [M][C] matrix, boxes of block_k channels x box_rows pixels.
cudaError_t tc_encode_x_matrix(const ConvProblem &p, int block_k, int box_rows, CUtensorMap *out);
cudaError_t tc_encode_w_tile(const ConvProblem &p, int block_k, int rows, CUtensorMap *out);
cudaError_t tc_encode_y_rows(const ConvProblem &p, const void *base, int box_c, int box_m, CUtensorMap *out);
// Dynamic shared memory of the tcgen05 kernel; `pair`: a 2-CTA pair holds half of each weight tile per CTA.
int tc_smem_bytes(int block_n, int block_k, int stages, int pair);

// Launchers; return cudaSuccess or the first CUDA error met.
cudaError_t tc_launch(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream);
// As tc_launch, but a stream-K plan uses `workspace` (plan.workspace_bytes long,
// its first plan.flag_bytes zeroed) instead of the library-held buffer; nullptr
// means the library-held buffer.
cudaError_t tc_launch_with_workspace(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream,
                                     void *workspace);
cudaError_t direct_launch(const ConvProblem &p, cudaStream_t stream);
// True when direct_launch has a fully unrolled variant for this filter shape.
bool direct_small_available(int r, int s, int c);
// Unfused comparator steps: t2 = BN(t1) and y = SiLU(t2), elementwise over NHWC bf16.
cudaError_t bn_apply_launch(const void *t1, const float *scale, const float *bias, void *t2, long long count,
                            int c_out, cudaStream_t stream);
cudaError_t silu_apply_launch(const void *t2, void *y, long long count, cudaStream_t stream);
// One layer of a batched BN fold (conv_bn_silu_fold_batch).
struct FoldLayer {
    const float *gamma, *beta, *mean, *var;
    float eps;
    int c_out;
    float *scale, *bias;
};
constexpr int kFoldBatchMax = 16;  // layers per launch (kernel parameter space)
struct FoldBatch {
    FoldLayer layer[kFoldBatchMax];
    int first_block[kFoldBatchMax];
    int count;
};
cudaError_t fold_batch_launch(const FoldLayer *layers, int count, cudaStream_t stream);
cudaError_t fold_launch(const float *gamma, const float *beta, const float *mean, const float *var,
                        float eps, int c_out, float *scale, float *bias, cudaStream_t stream);

// Thin-input tensor-core kernel (tc_gather.cu): 3x3 filters over 1, 3 or 4
// channels, at most 64 output channels.
bool gather_supported(const ConvProblem &p);
struct GatherPlan {
    int grid, tiles, block_n, block_k, stages, smem_bytes;
    int pass_rows;  // output rows per staging pass at most (a CTA's whole share when its rows fit at once)
};
// The thin-input kernel's launch for this shape on `sm_count` SMs; false when it cannot run it.
bool gather_plan(const ConvProblem &p, int sm_count, GatherPlan *out);
cudaError_t gather_launch(const ConvProblem &p, int sm_count, cudaStream_t stream);
cudaError_t gather_read_and_clear_error(cudaStream_t stream, unsigned int *out);
constexpr int kGatherBlockThreads = 288;

// Device error words (one per kernel translation unit): read and clear, stream-ordered.
cudaError_t tc_read_and_clear_error(cudaStream_t stream, unsigned int *out);
// Library-held stream-K workspaces: one per (device, stream), at most this many.
constexpr int kWorkspaceStreams = 64;
// Makes sure the current device and `stream` have an entry in the workspace table
// (created empty when missing); false when the table is full.
bool tc_workspace_reserve(cudaStream_t stream);
// Re-zeroes the stream-K ready flags of every workspace the library holds (after a
// kernel gave up mid-way, flags may be left raised).  Synchronous.
cudaError_t tc_reset_workspaces();

// Device error codes written by kernels (bit flags).
constexpr unsigned int kErrTimeoutProducer = 1u;
constexpr unsigned int kErrTimeoutMma = 2u;
constexpr unsigned int kErrTimeoutEpilogue = 4u;
constexpr unsigned int kErrTimeoutDrain = 8u;

}  // namespace cbs
