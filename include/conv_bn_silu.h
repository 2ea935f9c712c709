/*
 * conv_bn_silu.h -- C ABI of the fused conv2d -> BatchNorm -> SiLU layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer computes, per output pixel and output channel k,
 *
 *     y = SiLU(conv2d(x, W) * scale[k] + bias[k]),   SiLU(z) = z * sigmoid(z),
 *
 * as one kernel that reads x once and writes y once: the BatchNorm multiply/add
 * and the SiLU are applied to the convolution's output tile while it is still
 * on chip ("Fusing an Epilogue", kernels book, sections "The problem",
 * "What an epilogue is" and "The shape of it").
 *
 * Conventions shared by every entry point:
 *   - Layouts: x is NHWC [n][h][w][c] bf16; W is KRSC [c_out][r][s][c] bf16
 *     (for each output channel, the filter taps row by row, channels
 *     innermost); y is NHWC [n][ho][wo][c_out] bf16; every tensor dense.
 *   - The convolution is a cross-correlation with zero padding, dilation 1 and
 *     groups 1; ho = (h + 2*pad_h - r)/stride_h + 1 (floor), likewise wo.
 *   - Pointers named device are CUDA device (or managed) memory owned by the
 *     caller.  The library keeps no reference to them after a call returns and
 *     never frees or reallocates them.  Inputs are never written.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous: they validate, enqueue and return.
 *   - Every function returns a cbs_status.  Invalid arguments return an error
 *     without launching anything.  A fault inside a kernel surfaces at the
 *     caller's next synchronisation, like any CUDA launch; a pipeline wait
 *     that exceeded its time bound inside a kernel is reported by
 *     conv_bn_silu_check().
 *   - Thread safety: all entry points may be called from several host threads.
 */
#ifndef CONV_BN_SILU_H
#define CONV_BN_SILU_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cbs_status {
    CBS_OK = 0,
    CBS_ERR_INVALID_ARG = 1, /* null pointer, dim <= 0, stride < 1, pad < 0, ho/wo < 1, eps < 0 */
    CBS_ERR_MISALIGNED = 2,  /* a device pointer is not 16-byte aligned */
    CBS_ERR_UNSUPPORTED = 3, /* the requested algorithm cannot run this shape */
    CBS_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed; see conv_bn_silu_last_cuda_error() */
    CBS_ERR_TIMEOUT = 5      /* a kernel's pipeline wait ran past its bound and the kernel gave up */
} cbs_status;

/* Kernel choice for conv_bn_silu_forward_algo(). */
typedef enum cbs_algo {
    CBS_ALGO_AUTO = 0,    /* pick by shape (what conv_bn_silu_forward does) */
    CBS_ALGO_TCGEN05 = 1, /* implicit GEMM on the tcgen05 tensor cores, TMA-fed, TMEM accumulator */
    CBS_ALGO_DIRECT = 2   /* CUDA-core direct convolution, one output pixel per thread; any shape */
} cbs_algo;

/*
 * BatchNorm fold, run once per layer at load time.
 *   scale[k] = gamma[k] / sqrt(var[k] + eps),  bias[k] = beta[k] - mean[k] * scale[k]
 * The fusion page treats BN as one multiply and one add per element, with a
 * scale and a bias per output channel ("Fusing an Epilogue", sections "The
 * problem" and "The shape of it"); this is the inference-mode fold with running
 * statistics.  Computed in double precision, rounded once to float.
 *   gamma, beta, mean, var : device, float32 [c_out]
 *   eps                    : >= 0 and finite
 *   scale, bias            : device, float32 [c_out], written; must not overlap the inputs
 * c_out == 0 is a no-op.  var + eps <= 0 yields NaN/Inf in scale (not checked).
 */
int conv_bn_silu_fold(const float *gamma, const float *beta, const float *mean, const float *var,
                      float eps, int c_out, float *scale, float *bias, void *stream);

/*
 * The same fold for several layers in one launch (a network's layers at load
 * time, or every layer of a step): layer i's arguments and results are those
 * of conv_bn_silu_fold with layers[i]'s fields; the results are bit-identical.
 *   layers   : host array of n_layers descriptors, read during the call only
 *   n_layers : >= 0; 0 is a no-op.  Layers with c_out == 0 are skipped.
 * Every layer is validated before anything is launched (the first invalid
 * one decides the status).  Output arrays of different layers must not
 * overlap each other or any input.
 */
typedef struct cbs_fold_layer {
    const float *gamma, *beta, *mean, *var; /* device, float32 [c_out] */
    float eps;                              /* >= 0 and finite */
    int c_out;
    float *scale, *bias;                    /* device, float32 [c_out], written */
} cbs_fold_layer;

int conv_bn_silu_fold_batch(const cbs_fold_layer *layers, int n_layers, void *stream);

/*
 * Fused forward pass: y = SiLU(conv2d(x, W) * scale + bias).
 * ("Fusing an Epilogue", section "The shape of it": the K loop accumulates
 * the output tile; while it is still on chip, a per-channel multiply-add
 * and then SiLU are applied, and the tile is stored once; section "Three
 * kernels for one operation": convolution as a GEMM on the tensor cores.)
 *   x     : device, bf16 NHWC [n][h][w_in][c]
 *   w     : device, bf16 KRSC [c_out][r][s][c]
 *   scale : device, float32 [c_out]  (from conv_bn_silu_fold, or any per-channel multiplier)
 *   bias  : device, float32 [c_out]
 *   y     : device, bf16 NHWC [n][ho][wo][c_out], written; must not overlap x, w, scale or bias
 * All device pointers must be 16-byte aligned.  n == 0 or c_out == 0 is a
 * no-op.  The result is bf16 rounded to nearest even from an fp32
 * accumulator; it is deterministic (no atomics, fixed reduction order).
 * Kernels: the tcgen05 implicit GEMM when c % 16 == 0 and c_out % 8 == 0,
 * the thin-input tcgen05 kernel for 3x3 filters over 1, 3 or 4 channels,
 * otherwise the CUDA-core direct kernel.
 * Host work and memory held by the library, which this and every other
 * forward entry point (except conv_bn_silu_forward_noalloc) may do:
 *   - The first call of a shape on a set of buffers encodes TMA descriptors
 *     (host driver calls; cached for later calls), and the first launch of a
 *     kernel on a device sets its shared-memory limit.
 *   - Plans that split K loops between CTAs (cbs_plan_info.stream_k == 1,
 *     e.g. the 32x20x20x512 -> 512 3x3 layer) keep fp32 partial tiles in a
 *     scratch buffer the library holds, one per (device, stream).  The first
 *     such call on a stream allocates it with cudaMalloc (an implicit device
 *     synchronisation) and zeroes its flags with cudaMemsetAsync on `stream`;
 *     a later call that needs a larger buffer first synchronises `stream`,
 *     frees the old buffer and allocates a new one.  The buffers are kept
 *     until the process exits.  Make each such shape's first call on a stream
 *     before capturing that stream into a CUDA graph.
 *   - At most 64 (device, stream) pairs can hold such a buffer: a stream-K
 *     call on a 65th returns CBS_ERR_UNSUPPORTED (nothing is launched).
 *     conv_bn_silu_forward_noalloc needs none of this.
 */
int conv_bn_silu_forward(const void *x, const void *w, const float *scale, const float *bias,
                         void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                         int stride_h, int stride_w, int pad_h, int pad_w, void *stream);

/* As conv_bn_silu_forward, with the kernel chosen by `algo` (a cbs_algo).
 * Returns CBS_ERR_UNSUPPORTED when that kernel cannot run this shape. */
int conv_bn_silu_forward_algo(const void *x, const void *w, const float *scale, const float *bias,
                              void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                              int stride_h, int stride_w, int pad_h, int pad_w, int algo,
                              void *stream);

/*
 * Allocation-free variant of conv_bn_silu_forward (CBS_ALGO_AUTO), for callers
 * that may not allocate device memory: code running under a framework's own
 * caching allocator or a fixed memory budget, real-time loops where
 * cudaMalloc's implicit synchronisation is not acceptable, or hosts that hand
 * out only pre-sized buffers.  The fusion page has no counterpart to this; it
 * is a deployment convenience of this library.
 * Same arguments, layouts, results and errors as conv_bn_silu_forward, and
 * the same plan: where the plan splits K loops between CTAs (stream-K), the
 * partial tiles go to a fixed 20 MiB device array inside the library instead
 * of a library-allocated buffer, so the result is bit-identical to
 * conv_bn_silu_forward's.  A split that would need more than 20 MiB (see
 * cbs_plan_info.workspace_bytes; on a 152-SM GB300 every split fits) runs
 * whole tiles per CTA instead, which need no scratch: same values within the
 * layer's tolerance, not necessarily bit-identical.  Nothing is allocated by
 * any call, and no memory is held per stream.
 *   - The first call on a device looks up that array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call shares the one array per device and clears its ready flags
 *     first (an asynchronous memset on `stream`): calls whose kernels overlap
 *     on the GPU, e.g. on two streams, race and may produce wrong results.
 *     Serialise them on one stream.
 */
int conv_bn_silu_forward_noalloc(const void *x, const void *w, const float *scale, const float *bias,
                                 void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                                 int stride_h, int stride_w, int pad_h, int pad_w, void *stream);

/* Activation applied by conv_bn_act_forward after the BN multiply/add. */
typedef enum cbs_activation {
    CBS_ACT_SILU = 0,     /* z * sigmoid(z): the layer of conv_bn_silu_forward */
    CBS_ACT_IDENTITY = 1, /* z: BN (or a plain per-channel bias add) without activation */
    CBS_ACT_RELU = 2      /* max(z, 0) */
} cbs_activation;

/*
 * The fused layer with another epilogue.  "Fusing an Epilogue", section "What
 * an epilogue is": work that touches each output element once and needs no
 * neighbours (an activation, a bias add, a scaling) belongs in the epilogue of
 * the kernel that produced the element; a residual add of a tensor shaped like
 * y meets the same rule.
 *   y = act(conv2d(x, W) * scale + bias) [+ residual]
 * Arguments as conv_bn_silu_forward (the same kernels, chosen the same way), plus
 *   residual   : device, bf16 NHWC [n][ho][wo][c_out], or NULL for none; added
 *                after the activation, in fp32, before the one bf16 rounding.
 *                It may be y itself (an in-place add) but must not otherwise
 *                overlap y.  16-byte aligned.
 *   activation : a cbs_activation; anything else returns CBS_ERR_INVALID_ARG.
 * A plain per-channel bias (no BN) is scale = 1, bias = b with CBS_ACT_IDENTITY.
 * CBS_ACT_SILU with residual NULL computes exactly what conv_bn_silu_forward does.
 */
int conv_bn_act_forward(const void *x, const void *w, const float *scale, const float *bias,
                        const void *residual, void *y, int n, int h, int w_in, int c, int c_out, int r,
                        int s, int stride_h, int stride_w, int pad_h, int pad_w, int activation,
                        void *stream);

/*
 * conv_bn_act_forward with a narrower output: y is fp8 e4m3 (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; largest finite value 448, no infinities),
 * one byte per element, NHWC [n][ho][wo][c_out].  Each value is rounded once,
 * from the fp32 epilogue result to the nearest e4m3 (ties to even), saturating
 * to +-448 ("Fusing an Epilogue", section "What an epilogue is": casts to a
 * narrower dtype are epilogue work).  No residual.  The tensor-core path needs
 * c_out % 16 == 0 (16-byte rows) and takes the same tiles as the bf16 layer;
 * other shapes run on the direct kernel.
 */
int conv_bn_act_forward_fp8(const void *x, const void *w, const float *scale, const float *bias, void *y,
                            int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h, int stride_w,
                            int pad_h, int pad_w, int activation, void *stream);

/*
 * Unfused comparator: the same layer as the three-kernel sequence that the
 * fusion replaces -- the convolution writes t1 to memory, a BatchNorm kernel
 * reads t1 and writes t2, a SiLU kernel reads t2 and writes y ("Fusing an
 * Epilogue", kernels book, section "The problem": each step a round trip
 * through memory; section "When not to fuse": measure the fused kernel
 * against the sequence it replaces).  It exists to be measured against
 * conv_bn_silu_forward, not to be used in its place.
 *   t1 = bf16(conv2d(x, W))            (the forward kernel with the epilogue reduced to the cast)
 *   t2 = bf16(t1 * scale[k] + bias[k])
 *   y  = bf16(SiLU(t2))
 * Arguments as conv_bn_silu_forward, plus
 *   t1, t2 : device, bf16 NHWC [n][ho][wo][c_out] each, written (caller-owned
 *            scratch; must not overlap each other or any other argument)
 * y differs from conv_bn_silu_forward's by the two extra bf16 roundings of
 * t1 and t2.  Three kernels are enqueued on `stream`.
 */
int conv_bn_silu_forward_unfused(const void *x, const void *w, const float *scale, const float *bias,
                                 void *t1, void *t2, void *y, int n, int h, int w_in, int c, int c_out,
                                 int r, int s, int stride_h, int stride_w, int pad_h, int pad_w,
                                 void *stream);

/* The comparator's BatchNorm step on its own, over `count` bf16 elements of
 * an NHWC tensor with c_out channels (count % c_out == 0, count <= 2^40):
 *   t2[i] = bf16(t1[i] * scale[i mod c_out] + bias[i mod c_out]), fp32 arithmetic.
 * t1, t2: device bf16 [count]; scale, bias: device float32 [c_out]; all
 * 16-byte aligned; t2 must not overlap the inputs.  count == 0 is a no-op. */
int conv_bn_silu_bn_apply(const void *t1, const float *scale, const float *bias, void *t2,
                          long long count, int c_out, void *stream);

/* The comparator's SiLU step on its own: y[i] = bf16(SiLU(t2[i])) over `count`
 * bf16 elements (count <= 2^40), SiLU(z) = z * sigmoid(z) in fp32 ("Fusing
 * an Epilogue", section "The problem": SiLU is x times sigmoid of x).
 * t2, y: device bf16 [count], 16-byte aligned, not overlapping. */
int conv_bn_silu_silu_apply(const void *t2, void *y, long long count, void *stream);

/* Output spatial size of the convolution; host only, touches no GPU.
 * ho = (h + 2*pad_h - r)/stride_h + 1, wo likewise; CBS_ERR_INVALID_ARG when
 * either would be < 1 or an argument is out of range. */
int conv_bn_silu_output_dims(int h, int w_in, int r, int s, int stride_h, int stride_w,
                             int pad_h, int pad_w, int *ho, int *wo);

/* What conv_bn_silu_forward_algo would launch for this shape; host only. */
typedef struct cbs_plan_info {
    int algo;         /* cbs_algo actually selected (never CBS_ALGO_AUTO) */
    int block_m;      /* output pixels per tile */
    int block_n;      /* output channels per tile */
    int block_k;      /* reduction depth (channels) per pipeline stage */
    int stages;       /* shared-memory pipeline depth (0 for the direct kernel) */
    int tiles;        /* output tiles */
    int grid;         /* CTAs launched */
    int threads;      /* threads per CTA */
    int smem_bytes;   /* dynamic shared memory per CTA */
    int k_iters;      /* pipeline steps per tile */
    int stream_k;     /* 1 when the K steps of all tiles are split evenly over the grid */
    int swap_ab;      /* 1 when the GEMM runs transposed: channels on the MMA's M side, pixels on N */
    int cluster;      /* CTAs per cluster: 2 when CTA pairs run the 2-CTA MMA, each holding half of every weight tile */
    long long workspace_bytes; /* library-held scratch for stream-K partial tiles (0 if none) */
    int balanced;     /* swap_ab only: 1 when each CTA takes an equal run of 32-pixel chunks (units of at
                         most 256 pixels) instead of whole 256-pixel tiles */
    int weights_resident; /* swap_ab only: 1 when each CTA keeps its 128-channel weight tile in tensor
                             memory for the whole kernel and streams only x (units of block_m pixels) */
    int row_boxes;    /* swap_ab only: 1 when x is loaded in boxes of whole output rows (units of
                         block_m pixels = whole rows of one image) instead of im2col boxes */
} cbs_plan_info;

/* Fills `info` for the given shape, algorithm and SM count (sm_count > 0;
 * pass the device's multiprocessor count).  Host only, touches no GPU. */
int conv_bn_silu_plan(int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h,
                      int stride_w, int pad_h, int pad_w, int algo, int sm_count,
                      cbs_plan_info *info);

/*
 * Overrides of the planner's choices, for measuring the alternatives on a
 * given shape ("Fusing an Epilogue", section "Three kernels for one
 * operation": which kernel and tile run is a threshold somebody measures and
 * writes down).  -1 (block_n: 0) leaves that choice to the planner.
 */
typedef struct cbs_plan_request {
    int algo;     /* cbs_algo */
    int swap_ab;  /* -1, or 0: pixel-major tiles, 1: channel-major tiles (swap AB: 128 channels x 256 pixels) */
    int stream_k; /* -1, or 0: whole tiles per CTA, 1: K steps split evenly over the grid */
    int pair;     /* -1, or 0: single CTAs, 1: 2-CTA pairs (256-wide pixel-major tiles with stream-K only) */
    int block_n;  /* 0, or 16/32/64/128/256 output channels per pixel-major tile */
    long long wait_timeout_ns; /* 0: the default bound (2 s) on every pipeline wait of the tcgen05
                                  kernel; > 0: that bound instead.  A kernel whose wait runs out
                                  records it, stops, waits for its own copies in flight, frees its
                                  tensor memory and returns: conv_bn_silu_check then reports
                                  CBS_ERR_TIMEOUT, and later calls run normally.  (A bound of a
                                  few nanoseconds makes the waits run out on purpose: the watchdog
                                  test.)  Ignored by the other kernels. */
    int balanced; /* -1, or (channel-major tiles only) 0: whole 256-pixel tiles dealt round-robin,
                     1: each CTA an equal run of 32-pixel chunks */
    int weights_resident; /* -1, or 0: weights loaded with every tile, 1: the weight tile resident in
                             tensor memory (channel-major tiles, bf16 output without a residual, when
                             the tile fits next to two accumulators) */
    int row_boxes;        /* -1, or (channel-major tiles, bf16 output without a residual) 1: x loaded in
                             boxes of whole output rows (W divisible by the stride, equal strides, up
                             to 256 output columns), 0: im2col boxes */
} cbs_plan_request;

/* conv_bn_silu_plan with overrides.  CBS_ERR_INVALID_ARG for an out-of-range
 * field; CBS_ERR_UNSUPPORTED when the kernel cannot run the combination on
 * this shape (e.g. stream-K with shares shorter than one tile, pairs without
 * stream-K, any tcgen05 override on the thin-input or direct kernels). */
int conv_bn_silu_plan_request(int n, int h, int w_in, int c, int c_out, int r, int s, int stride_h,
                              int stride_w, int pad_h, int pad_w, const cbs_plan_request *req, int sm_count,
                              cbs_plan_info *info);

/* conv_bn_silu_forward_algo with overrides (req->algo replaces `algo`); the
 * same result within the layer's tolerance, whatever the tiling. */
int conv_bn_silu_forward_request(const void *x, const void *w, const float *scale, const float *bias,
                                 void *y, int n, int h, int w_in, int c, int c_out, int r, int s,
                                 int stride_h, int stride_w, int pad_h, int pad_w, const cbs_plan_request *req,
                                 void *stream);

/* Synchronises `stream`, then reads and clears the library's device error word.
 * Returns CBS_ERR_TIMEOUT if any kernel since the last check gave up on a
 * pipeline wait, CBS_ERR_CUDA if the synchronisation failed, else CBS_OK. */
int conv_bn_silu_check(void *stream);

/* Short English text for a cbs_status value (static storage, never NULL). */
const char *conv_bn_silu_status_string(int status);

/* The cudaError_t behind the calling thread's most recent CBS_ERR_CUDA (0 if none). */
int conv_bn_silu_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CONV_BN_SILU_H */
