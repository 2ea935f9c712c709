// tc_gather.cu -- fused conv2d + BatchNorm + SiLU on the tcgen05 tensor cores
// for thin inputs (3x3 filters over 1, 3 or 4 channels, e.g. a 3-channel stem),
// whose pixel rows are too narrow for TMA (a 6-byte pixel stride breaks its
// 16-byte stride rule).
//
// Same GEMM view as tc_conv.cu (M = output pixels, N = output channels,
// K = R*S*C ordered (r, s, c)), but the whole K fits one shared-memory row of
// KPAD = 32 or 64 bf16 (zero beyond R*S*C), so each 128-pixel tile is two or
// four MMAs.  The layer is bound by moving x and y, so the kernel is built
// around streaming them once:
//   - Each CTA owns one equal, contiguous range of output pixels (no ragged
//     last wave).  The input rows that range reads are one contiguous run of
//     NHWC memory (rows of consecutive images follow each other), and the
//     CTA copies that run into shared memory with a few cp.async.bulk
//     copies issued at its start, so each input row enters the SM once; the
//     few bytes of an unaligned head or tail are loaded with plain loads.
//     A range whose rows do not fit the staging buffer is cut into passes of
//     at most a few output rows each.
//   - warps 4..7  builders: one thread per pixel of a 128-pixel tile reads its
//                 receptive field from the staged rows (zeros in the padding)
//                 and writes its 64/128-byte row of the swizzled A stage;
//   - warp 8      MMA issuer: tcgen05.mma (M=128, N, K=16) against the weight
//                 tile B, resident in shared memory for the whole kernel;
//   - warps 0..3  epilogue: loads the weights and BN parameters while the
//                 input rows are in flight; per tile, tcgen05.ld of the
//                 accumulator, BN multiply/add, SiLU, bf16, and one contiguous
//                 2*N-byte store per pixel (a warp stores 32 consecutive
//                 pixels, i.e. consecutive rows of y).
// Every wait is bounded in time; on a timeout the kernel records an error bit,
// waits (bounded) for its own copies in flight, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {

__device__ unsigned int g_gather_error = 0;

namespace {

constexpr uint64_t kGatherTimeoutNs = 2000000000ull;
constexpr int kGatherThreads = kGatherBlockThreads;  // 4 epilogue + 4 builder warps + the MMA warp
constexpr int kGatherR = 3, kGatherS = 3;
constexpr int kStageCap = 32768;       // bytes of staged input rows per pass
constexpr int kStageSlack = 64;        // bytes after the staging buffer that tap reads may touch
constexpr int kBulkPiece = 16384;      // bytes per cp.async.bulk copy

struct GatherArgs {
    const __nv_bfloat16 *x;
    const __nv_bfloat16 *w;
    const float *scale;
    const float *bias;
    __nv_bfloat16 *y;
    long long m;         // output pixels
    int h, w_in, c_out, ho, wo, howo;
    int stride_h, stride_w, pad_h, pad_w;
    int row_bytes;       // bytes of one input row, w_in * C * 2
    int pass_rows;       // a staging pass ends at most this many output rows after its first row starts
    int epi_mode;        // EpiMode applied to the accumulator
    const __nv_bfloat16 *residual;  // nullable: bf16 [m][c_out] added after the activation
};

// CTAs resident per SM: three for 3 input channels (a 64-byte operand row: three CTAs' shared
// memory fits, and the kernel fits 75 registers a thread without spilling), two otherwise.
// More CTAs per SM means fewer 128-pixel tiles per CTA, whose A rows each CTA's builders
// write one tile after another.
__host__ __device__ constexpr int kGatherCtasPerSm(int c) { return c == 3 ? 3 : 2; }

template <int C, int N>
struct GatherCfg {
    static constexpr int TAPS = kGatherR * kGatherS * C;
    static constexpr int KPAD = TAPS <= 32 ? 32 : 64;
    static constexpr int ROW = KPAD * 2;                  // bytes per operand row = swizzle span
    static constexpr int STAGES = ROW == 64 ? 4 : 3;
    static constexpr int A_BYTES = 128 * ROW;
    static constexpr int B_BYTES = ((N * ROW + 1023) / 1024) * 1024;
    static constexpr int TMEM_COLS = 2 * N <= 32 ? 32 : (2 * N <= 64 ? 64 : 128);  // power of two
    static constexpr int SMEM = 1024 + STAGES * A_BYTES + B_BYTES + kStageCap + kStageSlack + 256;  // + barriers
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

// The global input rows that output pixels [p0, p1) read, as row indices of x
// viewed as [n*h][w_in*C] (consecutive images' rows are consecutive).  An
// empty range (first > last) when every tap of every pixel lies in the padding.
struct RowSpan {
    long long first, last;
};

// Pixel indices are below 2^31 (gather_supported), so the divisions are 32-bit.
__host__ __device__ inline RowSpan pass_rows(int p0, int p1, int howo, int wo, int h, int stride_h, int pad_h)
{
    const int ia = p0 / howo, ib = (p1 - 1) / howo;
    const int oha = (p0 - ia * howo) / wo, ohb = (p1 - 1 - ib * howo) / wo;
    const long long lo = (long long)oha * stride_h - pad_h, hi = (long long)ohb * stride_h - pad_h + kGatherR - 1;
    RowSpan r;
    r.first = (long long)ia * h + (lo < 0 ? 0 : lo);
    r.last = (long long)ib * h + (hi > h - 1 ? h - 1 : hi);
    return r;
}

// Byte layout of one pass's staged rows: global bytes [gs, ge) of x, placed in
// shared memory at offset (gs - a0), a0 = gs rounded down to 16, so that the
// 16-byte-aligned body [b0, b1) can be copied in bulk.
struct PassBytes {
    long long gs, ge, a0, b0, b1;
};

__host__ __device__ inline PassBytes pass_bytes(const RowSpan &rs, int row_bytes)
{
    PassBytes b;
    b.gs = rs.first * row_bytes;
    b.ge = rs.last >= rs.first ? (rs.last + 1) * row_bytes : b.gs;
    b.a0 = b.gs & ~15LL;
    b.b0 = (b.gs + 15) & ~15LL;
    b.b1 = b.ge & ~15LL;
    if (b.b1 < b.b0) b.b1 = b.b0;  // a run shorter than 16 bytes: all head
    return b;
}

// CTA b's share of m output pixels among g CTAs: the first m % g CTAs take one more
// (32-bit arithmetic only: m < 2^31).
__host__ __device__ inline void cta_share(int m, int b, int g, int *p0, int *p1)
{
    const int base = m / g, extra = m - base * g;
    *p0 = b * base + (b < extra ? b : extra);
    *p1 = *p0 + base + (b < extra ? 1 : 0);
}

// End of the staging pass that starts at output pixel ps: at most `pass_rows` output
// rows from the start of ps's row, and at most the CTA's share.
__host__ __device__ inline int pass_end(int ps, int p_end, int wo, int pass_rows)
{
    const long long e = (long long)(ps / wo + pass_rows) * wo;
    return e < p_end ? (int)e : p_end;
}

template <int C, int N>
__global__ void __launch_bounds__(kGatherThreads, kGatherCtasPerSm(C)) tc_gather_conv_bn_silu_kernel(const GatherArgs a)
{
    using G = GatherCfg<C, N>;
    constexpr int KPAD = G::KPAD;
    constexpr int ROW = G::ROW;
    constexpr int STAGES = G::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + STAGES * G::A_BYTES;
    uint8_t *sm_x = sm_b + G::B_BYTES;  // 1024-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_x + kStageCap + kStageSlack);
    uint64_t *full = bars;
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *xfull = drain + 1;    // a pass's staged rows have landed
    uint64_t *xempty = xfull + 1;   // every builder warp is done with a pass's staged rows
    uint64_t *bready = xempty + 1;  // the weight tile is in shared memory
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            dev::mbar_init(dev::smem_u32(&full[i]), 4);  // one arrival per builder warp
            dev::mbar_init(dev::smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&tfull[i]), 1);
            dev::mbar_init(dev::smem_u32(&tempty[i]), 4);
        }
        dev::mbar_init(dev::smem_u32(drain), 1);
        dev::mbar_init(dev::smem_u32(xfull), 1);
        dev::mbar_init(dev::smem_u32(xempty), 4);        // one arrival per builder warp
        dev::mbar_init(dev::smem_u32(bready), 4);        // one arrival per epilogue warp
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
    // This CTA's equal share of the output pixels, processed in passes of at most
    // pass_rows output rows (one pass when the share's input rows fit the staging buffer).
    // The share and the first pass's rows and bytes come from the launch arguments alone:
    // they are worked out before the wait for the preceding kernel, off the critical path.
    int p_begin, p_end;
    cta_share((int)a.m, (int)blockIdx.x, (int)gridDim.x, &p_begin, &p_end);
    const int pe_first = p_begin < p_end ? pass_end(p_begin, p_end, a.wo, a.pass_rows) : p_end;
    const RowSpan rs_first = pass_rows(p_begin, p_begin < p_end ? pe_first : p_begin + 1, a.howo, a.wo, a.h,
                                       a.stride_h, a.pad_h);
    const PassBytes pb_first = pass_bytes(rs_first, a.row_bytes);
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ builders
        const int row = (warp - 4) * 32 + lane;  // pixel of the tile this thread builds
        const int bt = threadIdx.x - 128;        // builder thread index, 0..127
        int stage = 0;
        uint32_t phase = 0;
        uint32_t xphase = 0;
        bool x_pending = false;  // a bulk copy of this CTA may still be in flight (issuing thread only)
        bool ok = true;
        const char *xg = reinterpret_cast<const char *>(a.x);
        int pass = 0;
        for (int ps = p_begin, pe; ps < p_end && ok; ps = pe, ++pass) {
            pe = pass == 0 ? pe_first : pass_end(ps, p_end, a.wo, a.pass_rows);
            const RowSpan rs = pass == 0 ? rs_first : pass_rows(ps, pe, a.howo, a.wo, a.h, a.stride_h, a.pad_h);
            const PassBytes pb = pass == 0 ? pb_first : pass_bytes(rs, a.row_bytes);
            if (warp == 4) {
                // Builder warp 4 stages the pass's rows, once every builder warp is done
                // reading the previous pass's: the unaligned head and tail (under 16 bytes
                // each, one 2-byte element per lane) with plain loads, then the
                // 16-byte-aligned body with bulk copies issued by lane 0.
                int okw = 1;
                if (lane == 0 && pass > 0)
                    okw = dev::mbar_wait_bounded(dev::smem_u32(xempty), (uint32_t)(pass - 1) & 1u, abort_flag,
                                                 kGatherTimeoutNs)
                              ? 1
                              : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    if (lane == 0 && !*abort_flag) gather_error(kErrTimeoutProducer, abort_flag);
                    ok = false;
                } else {
                    // The body's copies go out first (the barrier learns their byte count without
                    // an arrival); the head and tail loads, which wait for global memory, follow, and
                    // lane 0's arrival after the warp has stored them releases the whole pass.
                    const uint32_t xb = dev::smem_u32(xfull);
                    if (lane == 0) {
                        const long long body = pb.b1 - pb.b0;
                        if (body > 0) {
                            dev::mbar_expect_tx(xb, (uint32_t)body);
                            for (long long q = pb.b0; q < pb.b1; q += kBulkPiece) {
                                const uint32_t len = (uint32_t)(pb.b1 - q < kBulkPiece ? pb.b1 - q : kBulkPiece);
                                dev::bulk_load(dev::smem_u32(sm_x + (q - pb.a0)), xg + q, len, xb);
                            }
                            x_pending = true;
                        }
                    }
                    const long long head_end = pb.b0 < pb.ge ? pb.b0 : pb.ge;
                    const long long tail_beg = pb.b1 > head_end ? pb.b1 : head_end;
                    const int nhead = (int)((head_end - pb.gs) / 2), ntail = (int)((pb.ge - tail_beg) / 2);
                    const long long o = lane < nhead ? pb.gs + 2 * lane : tail_beg + 2 * (lane - 8);
                    if (lane < nhead || (lane >= 8 && lane - 8 < ntail))
                        dev::sts_u16(dev::smem_u32(sm_x) + (uint32_t)(o - pb.a0),
                                     __ldg(reinterpret_cast<const unsigned short *>(xg + o)));
                    __syncwarp();  // the plain writes happen before lane 0's arrive, which releases them
                    if (lane == 0) dev::mbar_arrive(xb);
                }
            }
            if (!dev::mbar_wait_bounded(dev::smem_u32(xfull), xphase, abort_flag, kGatherTimeoutNs)) {
                if (!*abort_flag) gather_error(kErrTimeoutProducer, abort_flag);
                ok = false;
                break;
            }
            xphase ^= 1u;
            if (bt == 0) x_pending = false;
            const uint32_t xs = dev::smem_u32(sm_x) + (uint32_t)(pb.gs - pb.a0);  // staged row `first` starts here
            for (int t0 = ps; t0 < pe; t0 += 128) {
                int okw = 1;
                if (lane == 0)
                    okw = dev::mbar_wait_bounded(dev::smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                                 kGatherTimeoutNs)
                              ? 1
                              : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    if (lane == 0 && !*abort_flag) gather_error(kErrTimeoutProducer, abort_flag);
                    ok = false;
                    break;
                }
                // This thread's receptive field, from the staged rows (zeros in the padding).
                // Pixel indices fit in 32 bits (m < 2^31); offsets into the staged rows are
                // below kStageCap.
                unsigned short v[G::TAPS];
                const int p = t0 + row;
                if (p < pe) {
                    const int img = p / a.howo;
                    const int rem = p - img * a.howo;
                    const int oh = rem / a.wo;
                    const int ow = rem - oh * a.wo;
                    // Staged row index of input row ih of this pixel's image: row0 + ih.
                    const int row0 = (int)((long long)img * a.h - rs.first);
                    // Input pixels iw0, iw0 + 1, iw0 + 2 of a row (the three taps s) are 6C
                    // contiguous bytes of the staged row: read as the aligned 32-bit words that
                    // cover them (two-byte aligned start: a funnel shift of 0 or 16 bits), a third
                    // of the load instructions of one two-byte load per value.  A tap in the
                    // padding reads neighbouring bytes (the weight tile before the staging buffer,
                    // the slack after it: at most 2 * 2C + 2 bytes before a row, 4 * NW after its
                    // last tap) and is zeroed below.
                    const int iw0 = ow * a.stride_w - a.pad_w;
                    bool cin[kGatherS];
#pragma unroll
                    for (int s = 0; s < kGatherS; ++s) cin[s] = iw0 + s >= 0 && iw0 + s < a.w_in;
                    constexpr int NW = (6 * C + 5) / 4;  // words covering 6C bytes from a two-byte offset
                    uint32_t in_mask = 0;
#pragma unroll
                    for (int r = 0; r < kGatherR; ++r) {
                        const int ih = oh * a.stride_h - a.pad_h + r;
                        const bool rin = ih >= 0 && ih < a.h;
                        const uint32_t start =
                            rin ? xs + (uint32_t)((row0 + ih) * a.row_bytes + iw0 * (C * 2)) : xs;
                        const uint32_t wa = start & ~3u, sh = (start & 2u) * 8u;
                        uint32_t w[NW];
#pragma unroll
                        for (int j = 0; j < NW; ++j) w[j] = dev::lds_u32(wa + 4u * j);
#pragma unroll
                        for (int s = 0; s < kGatherS; ++s) in_mask |= (rin && cin[s]) ? 1u << (r * kGatherS + s) : 0u;
#pragma unroll
                        for (int k = 0; k < kGatherS * C; ++k) {
                            const int j = k / 2, j1 = k / 2 + 1 < NW ? k / 2 + 1 : NW - 1;
                            const uint32_t two = __funnelshift_r(w[j], w[j1], sh);
                            v[r * kGatherS * C + k] = (unsigned short)((k & 1) ? two >> 16 : two & 0xffffu);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < G::TAPS; ++q)
                        if (!((in_mask >> (q / C)) & 1u)) v[q] = 0;
                } else {
#pragma unroll
                    for (int q = 0; q < G::TAPS; ++q) v[q] = 0;
                }
                const uint32_t arow = dev::smem_u32(sm_a) + (uint32_t)(stage * G::A_BYTES);
#pragma unroll
                for (int j = 0; j < ROW / 16; ++j) {
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = j * 8 + e * 2;
                        const uint32_t lo = q < G::TAPS ? v[q < G::TAPS ? q : 0] : 0u;
                        const uint32_t hi = q + 1 < G::TAPS ? v[q + 1 < G::TAPS ? q + 1 : 0] : 0u;
                        wv[e] = lo | (hi << 16);
                    }
                    dev::sts_v4(arow + swz<ROW>((uint32_t)(row * ROW + j * 16)), wv[0], wv[1], wv[2], wv[3]);
                }
                dev::fence_proxy_async_shared();  // generic-proxy writes -> tensor-core reads
                __syncwarp();
                if (lane == 0) dev::mbar_arrive(dev::smem_u32(&full[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(dev::smem_u32(xempty));  // this warp is done with the rows
        }
        // A copy still in flight (only after a wait gave up) must land before the CTA exits.
        if (x_pending && !dev::mbar_wait_bounded(dev::smem_u32(xfull), xphase, nullptr, kGatherTimeoutNs))
            gather_error(kErrTimeoutDrain, abort_flag);
    } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = dev::idesc_bf16_f32(128, N);
            const uint64_t desc_a0 = dev::smem_desc_kmajor(dev::smem_u32(sm_a), ROW);
            const uint64_t desc_b = dev::smem_desc_kmajor(dev::smem_u32(sm_b), ROW);
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            bool ok = dev::mbar_wait_bounded(dev::smem_u32(bready), 0, abort_flag, kGatherTimeoutNs);
            if (!ok && !*abort_flag) gather_error(kErrTimeoutMma, abort_flag);
            for (int ps = p_begin, pe; ps < p_end && ok; ps = pe) {
                pe = pass_end(ps, p_end, a.wo, a.pass_rows);
                for (int t0 = ps; t0 < pe; t0 += 128, ++lt) {
                    const int buf = lt & 1;
                    const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
                    if (!dev::mbar_wait_bounded(dev::smem_u32(&tempty[buf]), tparity ^ 1u, abort_flag,
                                                kGatherTimeoutNs) ||
                        !dev::mbar_wait_bounded(dev::smem_u32(&full[stage]), phase, abort_flag, kGatherTimeoutNs)) {
                        if (!*abort_flag) gather_error(kErrTimeoutMma, abort_flag);
                        ok = false;
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
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            dev::tc_commit(dev::smem_u32(drain));
            if (!dev::mbar_wait_bounded(dev::smem_u32(drain), 0, nullptr, kGatherTimeoutNs))
                gather_error(kErrTimeoutDrain, abort_flag);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ epilogue
        // Weight tile B first (while the input rows are in flight): row k = output
        // channel, K = (r, s, c) zero-padded to KPAD, in the swizzled K-major layout
        // the MMA descriptor describes.
        for (int i = threadIdx.x; i < N * (KPAD / 2); i += 128) {
            const int k = i / (KPAD / 2), q2 = (i - k * (KPAD / 2)) * 2;
            uint32_t lo = 0, hi = 0;
            if (k < a.c_out) {
                const unsigned short *wp = reinterpret_cast<const unsigned short *>(a.w) + (size_t)k * G::TAPS;
                if (q2 < G::TAPS) lo = __ldg(wp + q2);
                if (q2 + 1 < G::TAPS) hi = __ldg(wp + q2 + 1);
            }
            dev::sts_u32(dev::smem_u32(sm_b) + swz<ROW>((uint32_t)(k * ROW + q2 * 2)), lo | (hi << 16));
        }
        dev::fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(dev::smem_u32(bready));
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
        bool ok = true;
        for (int ps = p_begin, pe; ps < p_end && ok; ps = pe) {
            pe = pass_end(ps, p_end, a.wo, a.pass_rows);
            for (int t0 = ps; t0 < pe; t0 += 128, ++lt) {
                const int buf = lt & 1;
                const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
                int okw = 1;
                if (lane == 0)
                    okw = dev::mbar_wait_bounded(dev::smem_u32(&tfull[buf]), tparity, abort_flag, kGatherTimeoutNs)
                              ? 1
                              : 0;
                okw = __shfl_sync(0xffffffffu, okw, 0);
                if (!okw) {
                    if (lane == 0 && !*abort_flag) gather_error(kErrTimeoutEpilogue, abort_flag);
                    ok = false;
                    break;
                }
                dev::tc_fence_after_sync();
                // 16 columns (channels) at a time, so wide tiles keep few registers live; the
                // accumulator goes back to the MMA warp after its last columns are read.
                const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * N);
                const int m = t0 + warp * 32 + lane;
                const bool store = m < pe;
                const long long yoff = (long long)(store ? m : 0) * a.c_out;
                __nv_bfloat16 *yp = a.y + yoff;
                const __nv_bfloat16 *rp = a.residual != nullptr ? a.residual + yoff : nullptr;
#pragma unroll
                for (int q = 0; q < N / 16; ++q) {
                    uint32_t v[16];
                    dev::tmem_ld_32x32b_x16(taddr + (uint32_t)(q * 16), v);
                    dev::tmem_ld_wait();
                    dev::reg_fence16(v);
                    if (q == N / 16 - 1) {
                        dev::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                    }
                    if (!store) continue;
                    uint32_t packed[8];
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        const int j = q * 16 + jj;
                        float f0 = dev::epilogue_from_half(__uint_as_float(v[jj]), half_scale(j), half_bias(j), a.epi_mode);
                        float f1 = dev::epilogue_from_half(__uint_as_float(v[jj + 1]), half_scale(j + 1),
                                                           half_bias(j + 1), a.epi_mode);
                        if (rp != nullptr) {
                            f0 += j < a.c_out ? __bfloat162float(rp[j]) : 0.f;
                            f1 += j + 1 < a.c_out ? __bfloat162float(rp[j + 1]) : 0.f;
                        }
                        packed[jj / 2] = dev::pack_bf16x2(f0, f1);
                    }
                    if (a.c_out == N) {
                        uint4 *dst = reinterpret_cast<uint4 *>(yp + q * 16);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    } else {
                        unsigned short *d16 = reinterpret_cast<unsigned short *>(yp);
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj)
                            if (q * 16 + jj < a.c_out)
                                d16[q * 16 + jj] = (unsigned short)(packed[jj / 2] >> (16 * (jj & 1)));
                    }
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

// Output rows per staging pass: the largest k such that no pass of any CTA (at most k
// output rows from the start of its first row) needs more than kStageCap bytes of
// staged input rows.  k = 1 (a pass within one output row, never across images)
// always fits once gather_supported holds; 0 only if it does not.
int choose_pass_rows(const ConvProblem &p, int grid, int row_bytes)
{
    const long long howo = (long long)p.ho * p.wo;
    auto fits = [&](int k) {
        for (int b = 0; b < grid; ++b) {
            int p0, p1;
            cta_share((int)p.m, b, grid, &p0, &p1);
            for (int ps = p0, pe; ps < p1; ps = pe) {
                pe = pass_end(ps, p1, p.wo, k);
                const RowSpan rs = pass_rows(ps, pe, (int)howo, p.wo, p.h, p.stride_h, p.pad_h);
                const PassBytes pb = pass_bytes(rs, row_bytes);
                if (pb.ge - pb.a0 > kStageCap) return false;
            }
        }
        return true;
    };
    // Start from the rows one CTA's share covers (plus one for a share that starts mid-row).
    const long long share = (p.m + grid - 1) / grid;
    int k = (int)std::min<long long>(share / p.wo + 2, 1 << 20);
    const int by_cap = (kStageCap / row_bytes - kGatherR) / (p.stride_h > 0 ? p.stride_h : 1) + 1;
    k = std::max(1, std::min(k, by_cap));
    for (; k >= 1; --k)
        if (fits(k)) return k;
    return 0;
}

int gather_n(int c_out) { return c_out <= 16 ? 16 : (c_out <= 32 ? 32 : (c_out <= 48 ? 48 : 64)); }

template <int C, int N>
cudaError_t launch_gather(const ConvProblem &p, int grid, int pass_rows, cudaStream_t stream)
{
    using G = GatherCfg<C, N>;
    auto kern = tc_gather_conv_bn_silu_kernel<C, N>;
    static std::mutex mu;
    static unsigned long long done = 0;
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long bit = device < 64 ? (1ull << device) : 0ull;
        if (!(done & bit) || bit == 0) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (err != cudaSuccess) return err;
            done |= bit;
        }
    }
    GatherArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(p.x);
    a.w = static_cast<const __nv_bfloat16 *>(p.w);
    a.scale = p.scale;
    a.bias = p.bias;
    a.y = static_cast<__nv_bfloat16 *>(p.y);
    a.m = p.m;
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
    a.row_bytes = p.w_in * C * 2;
    a.pass_rows = pass_rows;
    a.epi_mode = p.epi_mode;
    a.residual = static_cast<const __nv_bfloat16 *>(p.residual);
    return launch_overlapped(kern, dim3((unsigned)grid), dim3(kGatherThreads), (size_t)G::SMEM, stream, 1, a);
}

template <int C>
cudaError_t launch_gather_c(const ConvProblem &p, int grid, int pass_rows, cudaStream_t stream)
{
    switch (gather_n(p.c_out)) {
    case 16: return launch_gather<C, 16>(p, grid, pass_rows, stream);
    case 32: return launch_gather<C, 32>(p, grid, pass_rows, stream);
    case 48: return launch_gather<C, 48>(p, grid, pass_rows, stream);
    default: return launch_gather<C, 64>(p, grid, pass_rows, stream);
    }
}

}  // namespace

bool gather_supported(const ConvProblem &p)
{
    if (p.m > 0x7fffffffLL - 128) return false;
    if (p.out_fp8) return false;  // the bf16 output only (the direct kernel writes fp8)
    // Padding of at most filter - 1: every output row reads at least one input row, which the
    // pass bounds (pass_rows) rely on, and the tap reads stay within the staging slack.
    const bool shape = p.r == kGatherR && p.s == kGatherS && (p.c == 1 || p.c == 3 || p.c == 4) &&
                       p.pad_h >= 0 && p.pad_h <= kGatherR - 1 && p.pad_w >= 0 && p.pad_w <= kGatherS - 1;
    if (!shape || p.c_out < 1 || p.c_out > 64) return false;
    // A single output pixel's rows must fit the staging buffer.
    return (long long)kGatherR * p.w_in * p.c * 2 + 32 <= kStageCap;
}

bool gather_plan(const ConvProblem &p, int sm_count, GatherPlan *out)
{
    if (!gather_supported(p)) return false;
    const long long tiles = (p.m + 127) / 128;
    const int grid = (int)std::min<long long>(tiles, (long long)kGatherCtasPerSm(p.c) * sm_count);
    // The pass size walks every CTA's passes once per shape; later calls hit this cache.
    struct Entry {
        long long m;
        int h, w_in, c, ho, wo, stride_h, pad_h, grid;
        int pass;
    };
    static std::mutex mu;
    static Entry cache[16];
    static int used = 0, next = 0;
    const Entry key{p.m, p.h, p.w_in, p.c, p.ho, p.wo, p.stride_h, p.pad_h, grid, 0};
    int pass = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry &e = cache[i];
            if (e.m == key.m && e.h == key.h && e.w_in == key.w_in && e.c == key.c && e.ho == key.ho &&
                e.wo == key.wo && e.stride_h == key.stride_h && e.pad_h == key.pad_h && e.grid == key.grid)
                pass = e.pass;
        }
    }
    if (pass < 0) {
        pass = choose_pass_rows(p, grid, p.w_in * p.c * 2);
        std::lock_guard<std::mutex> lock(mu);
        Entry e = key;
        e.pass = pass;
        cache[next] = e;
        next = (next + 1) % 16;
        if (used < 16) ++used;
    }
    if (pass <= 0) return false;
    const int taps = kGatherR * kGatherS * p.c;
    const int kpad = taps <= 32 ? 32 : 64;
    const int n = gather_n(p.c_out);
    const int stages = kpad == 32 ? 4 : 3;
    out->grid = grid;
    out->tiles = (int)tiles;
    out->pass_rows = pass;
    out->block_n = n;
    out->block_k = kpad;
    out->stages = stages;
    out->smem_bytes =
        1024 + stages * 128 * kpad * 2 + (n * kpad * 2 + 1023) / 1024 * 1024 + kStageCap + kStageSlack + 256;
    return true;
}

cudaError_t gather_launch(const ConvProblem &p, int sm_count, cudaStream_t stream)
{
    GatherPlan g{};
    if (!gather_plan(p, sm_count, &g)) return cudaErrorInvalidConfiguration;
    switch (p.c) {
    case 1: return launch_gather_c<1>(p, g.grid, g.pass_rows, stream);
    case 3: return launch_gather_c<3>(p, g.grid, g.pass_rows, stream);
    case 4: return launch_gather_c<4>(p, g.grid, g.pass_rows, stream);
    default: return cudaErrorInvalidConfiguration;
    }
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
