// tc_conv.cu -- fused conv2d + BatchNorm + SiLU as an implicit GEMM on the
// sm_103a tensor cores.
//
// GEMM view ("Fusing an Epilogue", kernels book, section "Three kernels for
// one operation": convolution as a GEMM on the tensor cores):
//   M = n*ho*wo output pixels, N = c_out, K = r*s*c, laid out (r, s, c) so that
//   the KRSC weight tensor is already the K-major B operand (the K steps, one
//   tap x BK channels each, are visited with the taps running fastest).
//   A[m][k] = x[img][oh*sh - ph + r][ow*sw - pw + s][c], zero outside the image.
//
// Per CTA (one per SM, persistent over output tiles of 128 pixels x BN channels):
//   warp 0      TMA producer: per K step, one im2col load of A (128 pixels x
//               BK channels of one filter tap, zero-filled at the borders) and
//               one tiled load of B (BN output channels x BK channels of that
//               tap) into a STAGES-deep shared-memory ring; no im2col buffer
//               ever exists in global memory.
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into a TMEM
//               accumulator; two accumulators so the epilogue of tile i
//               overlaps the K loop of tile i+1.
//   warps 4..   epilogue ("The shape of it"): tcgen05.ld of the finished tile
//               (warps w, w+4, ... share TMEM lanes 32*(w%4).. and split the
//               columns: two per lane quarter from 64 channels, three on the
//               2-CTA pair tiles, whose last tile's epilogue has no K loop
//               under it), acc*scale + bias, SiLU, bf16 cast, staged through
//               swizzled shared memory and written by TMA stores.  x is read once and y
//               written once; the conv result never goes to memory.
// Every mbarrier wait is bounded in time; on timeout the kernel records an
// error bit, waits for its own copies in flight, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "cbs_internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace cbs {

__device__ unsigned int g_tc_error = 0;

namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct TcArgs {
    const float *scale;
    const float *bias;
    int c_out;
    int m;  // output pixels
    int n_tiles, tiles;
    int howo, wo;
    int stride_h, stride_w, pad_h, pad_w;
    int s;
    int c_chunks, k_iters;
    int epi_mode;    // EpiMode applied to the accumulator
    const __nv_bfloat16 *residual;  // nullable: bf16 [m][c_out] added after the activation
    int stream_k;    // 1: each CTA takes an equal share of all K steps (see WorkIter)
    unsigned long long wait_ns;  // bound on every pipeline wait (draining copies in flight keeps 2 s)
    float *partial;  // stream-K: [grid-1][128*BN] fp32 partial tiles (slot c: boundary of CTAs c, c+1)
    int *flags;      // stream-K: per slot, a ready flag per (lane quarter, 32-column chunk); 0 between launches
    int balanced;    // swap AB: each CTA takes an equal run of 32-pixel chunks (see WorkIter)
    int chunks_m;    // balanced: 32-pixel chunks per channel tile, ceil(m / 32)
};

// K steps [kb, ke) of output tile `tile`.  Balanced channel-major units: `tile`
// is the channel tile and the unit covers pixels [p0, p0 + np).
struct WorkUnit {
    int tile, kb, ke;
    int p0, np;
};

// The units one worker processes.  A worker is a CTA, or a CTA pair sharing
// one weight tile (PAIR).  Data-parallel: whole tiles vb, vb + vg, ...
// Stream-K: the worker's equal share of the
// global K-step sequence (tile-major), cut at tile boundaries.  The host enables
// stream-K only when every share is at least one tile long, so a unit is a whole
// tile, the tail of a tile (kb > 0: the previous CTA holds its head) or the head
// of a tile (ke < k_iters: the next CTA holds its tail), never a middle piece.
struct WorkIter {
    // stream-K state: the worker's range is [tail piece][whole tiles][head piece];
    // it is processed as head, tail, then whole tiles (see next()).
    int state;
    int t_tail, kb_tail;   // tail piece: K steps [kb_tail, k_iters) of tile t_tail (kb_tail > 0)
    int t_head, ke_head;   // head piece: K steps [0, ke_head) of tile t_head (ke_head < k_iters)
    int t_full, t_full_end;  // whole tiles [t_full, t_full_end)
    // data-parallel state
    int t, stride;
    // balanced channel-major state: chunks [g, g1) of the (channel tile, 32-pixel chunk)
    // sequence, channel tile major.
    int g, g1;
    // vb / vg: this worker's index and the worker count (a CTA, or a CTA pair).
    // The host enables balanced runs and stream-K only when the sequence length times
    // the worker count fits in 32 bits, so the splits below use 32-bit divisions
    // (64-bit ones would delay every CTA's first load by hundreds of cycles).
    __device__ WorkIter(const TcArgs &a, int vb, int vg)
    {
        state = 0;
        t = vb;
        stride = vg;
        if (a.balanced) {
            const uint32_t total = (uint32_t)a.n_tiles * (uint32_t)a.chunks_m;
            g = (int)(total * (uint32_t)vb / (uint32_t)vg);
            g1 = (int)(total * (uint32_t)(vb + 1) / (uint32_t)vg);
        }
        if (a.stream_k) {
            const uint32_t total = (uint32_t)a.tiles * (uint32_t)a.k_iters;
            const uint32_t g0 = total * (uint32_t)vb / (uint32_t)vg, g1 = total * (uint32_t)(vb + 1) / (uint32_t)vg;
            const uint32_t ki = (uint32_t)a.k_iters;
            const int t0 = (int)(g0 / ki);
            const int kb0 = (int)(g0 - (uint32_t)t0 * ki);
            const int t1 = (int)((g1 - 1) / ki);
            const int ke1 = (int)(g1 - (uint32_t)t1 * ki);
            t_tail = kb0 > 0 ? t0 : -1;
            kb_tail = kb0;
            t_head = ke1 < a.k_iters ? t1 : -1;
            ke_head = ke1;
            t_full = kb0 > 0 ? t0 + 1 : t0;
            t_full_end = ke1 < a.k_iters ? t1 : t1 + 1;
        }
    }
    // Stream-K order: the head piece first, then the tail piece, then whole tiles.
    // Every worker starts at K step 0 of a tile, so the first stages of all CTAs
    // load the same weight tiles (from a cold L2 the start otherwise pulls most of
    // the weights at once); the split pieces meet their other halves (published
    // first by the neighbouring workers) mid-kernel, and the last epilogue of a
    // worker with whole tiles is a plain one.
    __device__ bool next(const TcArgs &a, WorkUnit &u)
    {
        if (a.balanced) {
            // Within one channel tile the worker's chunks are cut into units of 256
            // pixels (two whole im2col boxes) and one shorter remainder, so that no
            // box is loaded for fewer pixels than it holds except in the remainder.
            if (g >= g1) return false;
            const int nt = g / a.chunks_m;
            const int piece_end = g1 < (nt + 1) * a.chunks_m ? g1 : (nt + 1) * a.chunks_m;
            const int take = piece_end - g < 8 ? piece_end - g : 8;
            u.tile = nt;
            u.p0 = (g - nt * a.chunks_m) * 32;
            u.np = a.m - u.p0 < take * 32 ? a.m - u.p0 : take * 32;
            u.kb = 0;
            u.ke = a.k_iters;
            g += take;
            return true;
        }
        if (a.stream_k) {
            if (state == 0) {
                state = 1;
                if (t_head >= 0) {
                    u.tile = t_head;
                    u.kb = 0;
                    u.ke = ke_head;
                    return true;
                }
            }
            if (state == 1) {
                state = 2;
                if (t_tail >= 0) {
                    u.tile = t_tail;
                    u.kb = kb_tail;
                    u.ke = a.k_iters;
                    return true;
                }
            }
            if (t_full >= t_full_end) return false;
            u.tile = t_full++;
            u.kb = 0;
            u.ke = a.k_iters;
            return true;
        }
        if (t >= a.tiles) return false;
        u.tile = t;
        u.kb = 0;
        u.ke = a.k_iters;
        t += stride;
        return true;
    }
};

__device__ __forceinline__ int ld_acquire_gpu(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int *p, int v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait for another CTA's flag (both CTAs are resident: the grid never
// exceeds one CTA per SM).  False on timeout or when this CTA is aborting.
__device__ __forceinline__ bool wait_flag_bounded(const int *flag, const volatile int *abort_flag,
                                                  uint64_t timeout_ns)
{
    if (ld_acquire_gpu(flag) != 0) return true;
    const uint64_t t0 = dev::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ld_acquire_gpu(flag) != 0) return true;
        if ((i & 15u) == 0) {
            if (*abort_flag) return false;
            if (dev::globaltimer_ns() - t0 > timeout_ns) return false;
        }
        __nanosleep(64);
    }
}

// B_ROWS: weight (B) rows held per CTA -- BN, or BN/2 when a CTA pair splits them.
template <int BN, int BK, int B_ROWS = BN, bool PAIRED = false>
struct TcCfg {
    static constexpr int BM = kTcBlockM;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = B_ROWS * BK * 2;
    static constexpr int A_STRIDE = (A_BYTES + 1023) / 1024 * 1024;
    static constexpr int B_STRIDE = (B_BYTES + 1023) / 1024 * 1024;
    static constexpr int SPLIT = BN >= 64 ? 2 : 1;  // sets the chunk width below
    static constexpr int EC = BN / SPLIT < 32 ? BN / SPLIT : 32;  // epilogue columns per chunk
    static constexpr int NCH = BN / EC;                          // chunks across the tile
    // Epilogue warps per TMEM lane quarter; warp h of a quarter takes the chunks
    // [h * NCH / WPQ, (h + 1) * NCH / WPQ), at most MAX_OWN of them.
    static constexpr int WPQ = tc_epi_warps_per_quarter(BN, PAIRED);
    static constexpr int MAX_OWN = (NCH + WPQ - 1) / WPQ;
    static constexpr int EPI_WARPS = 4 * WPQ;
    static constexpr int THREADS = tc_threads(BN, PAIRED);
    static constexpr int STG_BYTES = 32 * EC * 2;  // one warp's staging buffer (32 rows)
    static constexpr int STG_TOTAL = EPI_WARPS * 2 * STG_BYTES;
    static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : 2 * BN;
    static constexpr int ROW_A = BK * 2;  // operand row bytes = swizzle span
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int BAR_BYTES = 512;
    static constexpr int STAGES_FIT =
        (SMEM_LIMIT - 1024 - STG_TOTAL - BAR_BYTES) / (A_STRIDE + B_STRIDE);
    static constexpr int STAGES = STAGES_FIT < 8 ? STAGES_FIT : 8;
    static constexpr int SMEM = 1024 + STAGES * (A_STRIDE + B_STRIDE) + STG_TOTAL + BAR_BYTES;
    static_assert(STAGES >= 2, "shared memory too small for two stages");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M=128");
    static_assert(BN % EC == 0 && NCH >= WPQ, "every epilogue warp owns at least one whole chunk");
    static_assert(4 * NCH <= kTcFlagsPerSlot && THREADS == 128 + 32 * EPI_WARPS, "epilogue warps");
    static_assert((2 * STAGES + 6 + 2 * EPI_WARPS) * 8 + 8 <= BAR_BYTES, "barrier area");
    static_assert(TMEM_COLS == 32 || TMEM_COLS == 64 || TMEM_COLS == 128 || TMEM_COLS == 256 ||
                      TMEM_COLS == 512,
                  "TMEM allocation must be a power of two >= 32");
};

__device__ __forceinline__ void record_error(unsigned int bit, volatile int *abort_flag)
{
    atomicOr(&g_tc_error, bit);
    *abort_flag = 1;
}

// XOR swizzle of a byte offset inside a 1024-byte aligned buffer whose rows
// are `ROW` bytes (32/64/128), matching CU_TENSOR_MAP_SWIZZLE_{32,64,128}B.
template <int ROW>
__device__ __forceinline__ uint32_t swizzle_offset(uint32_t off)
{
    constexpr uint32_t mask = ROW == 128 ? 7u : (ROW == 64 ? 3u : 1u);
    return off ^ (((off >> 7) & mask) << 4);
}

// SWAP = false: D[pixel][channel], A = im2col tile (128 pixels), B = weights (BN channels).
// SWAP = true ("swap AB", for C_out <= 128): D[channel][pixel], A = weights (128
// channels), B = im2col tile (BN = 256 pixels as two 128-pixel boxes), so the MMA
// runs at N = 256 -- with operands streamed from shared memory an M=128 MMA costs
// about the same time at N = 128 as at N = 256.  The epilogue transposes through
// shared memory.
// PAIR: the grid is launched as clusters of two CTAs that work as one on a
// 256 x BN pair tile with the 2-CTA tensor-core MMA (tcgen05 cta_group::2,
// M = 256): each CTA loads the A tile of its own 128 pixels and one half of
// the weight tile (BN/2 channels), and holds the 128 x BN accumulator of its
// pixels in its own TMEM.  Only the even CTA issues MMAs; the hardware feeds
// both tensor cores from both CTAs' shared memory.  Per K step a CTA takes in
// A + B/2 instead of A + B, and the smaller stages leave room for more of
// them.  Both CTAs' loads complete on the even CTA's full barrier; its MMA
// commits release the stage, and publish a finished accumulator, in both CTAs;
// both CTAs' epilogue warps hand the accumulator back to the even CTA.
// EPI: which epilogue the instantiation carries, so that the fused layer's own
// (BN + SiLU) pays nothing for the others -- kEpiKindSilu, kEpiKindMode (the
// launch's EpiMode, chosen at run time) or kEpiKindResidual (the same, plus a
// residual tensor added after the activation).
constexpr int kEpiKindSilu = 0;
constexpr int kEpiKindMode = 1;
constexpr int kEpiKindResidual = 2;
constexpr int kEpiKindFp8 = 3;  // the launch's EpiMode with an fp8 e4m3 output (pixel-major tiles only)

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_l1(const void *p)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Calls f(std::integral_constant<int, mode>) with the epilogue mode as a compile-time
// constant: SiLU alone for the fused layer's instantiation, else one arm per mode.
template <int EPI, typename F>
__device__ __forceinline__ void with_epi_mode(int mode, F &&f)
{
    if constexpr (EPI == kEpiKindSilu) {
        f(std::integral_constant<int, kEpiSilu>{});
    } else {
        switch (mode) {
        case kEpiConvOnly: f(std::integral_constant<int, kEpiConvOnly>{}); break;
        case kEpiBn: f(std::integral_constant<int, kEpiBn>{}); break;
        case kEpiRelu: f(std::integral_constant<int, kEpiRelu>{}); break;
        default: f(std::integral_constant<int, kEpiSilu>{}); break;
        }
    }
}

template <int BN, int BK, bool SWAP, bool PAIR, int EPI>
__global__ void __launch_bounds__(TcCfg<BN, BK, PAIR ? BN / 2 : BN, PAIR>::THREADS, 1)
    tc_conv_bn_silu_kernel(const __grid_constant__ CUtensorMap tm_x,
                           const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_y,
                           const __grid_constant__ CUtensorMap tm_r, const TcArgs a)
{
    static_assert(!(SWAP && PAIR), "CTA pairs serve the pixel-major (unswapped) tile only");
    static_assert(!SWAP || TcCfg<BN, BK>::EC == 32, "channel-major units are cut in 32-pixel chunks");
    constexpr bool RES = EPI == kEpiKindResidual;
    constexpr bool FP8 = EPI == kEpiKindFp8;
    // The epilogue mode: a compile-time constant for the fused layer.
    const int emode = EPI == kEpiKindSilu ? (int)kEpiSilu : a.epi_mode;
    constexpr int CG = PAIR ? 2 : 1;  // tcgen05 CTA group
    using C = TcCfg<BN, BK, PAIR ? BN / 2 : BN, PAIR>;
    constexpr int STAGES = C::STAGES;
    // Pair tiles: the four warps that load and issue (0-3) have nothing left to do once a
    // worker's last unit is in TMEM, and join its epilogue as a fourth warp per TMEM lane
    // quarter (the last tile's epilogue has no K loop under it).  Not with a residual, whose
    // loads use a barrier per staging buffer of the epilogue warps.
    constexpr bool HELP = PAIR && !RES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sm_a = smem;
    uint8_t *sm_b = sm_a + STAGES * C::A_STRIDE;
    uint8_t *sm_stg = sm_b + STAGES * C::B_STRIDE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm_stg + C::STG_TOTAL);
    uint64_t *full = bars;
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *lastfull = drain + 1;  // pair tiles: the worker's last MMA is done (helpers wait on it)
    uint64_t *rbar = lastfull + 1;  // residual epilogue: a load barrier per staging buffer of each epilogue warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(rbar + 2 * C::EPI_WARPS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = PAIR ? (int)dev::cluster_ctarank() : 0;  // M half of the pair tile
    const int vb = PAIR ? (int)blockIdx.x >> 1 : (int)blockIdx.x;
    const int vg = PAIR ? (int)gridDim.x >> 1 : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            dev::mbar_init(dev::smem_u32(&full[i]), 2);  // the two producers' arrivals
            dev::mbar_init(dev::smem_u32(&empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            dev::mbar_init(dev::smem_u32(&tfull[i]), 1);
            // A pair's accumulator is released by the epilogue warps of both CTAs.
            dev::mbar_init(dev::smem_u32(&tempty[i]), PAIR ? 2 * C::EPI_WARPS : C::EPI_WARPS);
        }
        dev::mbar_init(dev::smem_u32(drain), 1);
        dev::mbar_init(dev::smem_u32(lastfull), 1);
        if constexpr (RES)
            for (int i = 0; i < 2 * C::EPI_WARPS; ++i) dev::mbar_init(dev::smem_u32(&rbar[i]), 1);
        *abort_flag = 0;
        dev::fence_mbarrier_init();
    }
    if (threadIdx.x == 32) {
        dev::prefetch_tensormap(&tm_x);
        dev::prefetch_tensormap(&tm_w);
        dev::prefetch_tensormap(&tm_y);
        if constexpr (RES) dev::prefetch_tensormap(&tm_r);
    }
    if (warp == 1) {
        // CG = 2: collective over the pair (warp 1 of both CTAs); same columns in both.
        dev::tmem_alloc<CG>(dev::smem_u32(tmem_slot), C::TMEM_COLS);
        dev::tmem_relinquish_alloc_permit<CG>();
    }
    dev::tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) dev::cluster_sync();  // the peer's barriers exist before any remote signal
    dev::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // PAIR: the even CTA's barriers that both CTAs signal, as shared::cluster addresses.
    const uint32_t full0 = PAIR ? dev::mapa_cluster(dev::smem_u32(full), 0) : 0u;
    const uint32_t tempty0 = PAIR ? dev::mapa_cluster(dev::smem_u32(tempty), 0) : 0u;
    // Global memory is touched only after the preceding kernel has finished.
    dev::grid_dependency_wait();
    dev::grid_dependents_launch();

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        // Two issuing threads: warp 0 loads the x operand (im2col boxes), warp 2 the weight
        // tile; each arrives on the stage's full barrier with its own byte count.  One thread
        // issuing every box left the loads short of what the tensor pipe consumes.
        const bool loads_w = warp == 2;
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_parity = 0;
            WorkIter wi(a, vb, vg);
            WorkUnit u;
            while (!*abort_flag && wi.next(a, u)) {
                const int m_unit = u.tile / a.n_tiles;
                const int m_tile = PAIR ? 2 * m_unit + rank : m_unit;
                const bool bal = SWAP && a.balanced;
                const int n0 = bal ? u.tile * C::BM : (u.tile - m_unit * a.n_tiles) * (SWAP ? C::BM : BN);
                const int m0 = bal ? u.p0 : m_tile * (SWAP ? BN : C::BM);  // first pixel
                // SWAP: one 128-pixel box, or two when the unit has more pixels than one holds.
                const bool two_boxes = !bal || u.np > C::BM;
                const int img = m0 / a.howo;
                const int rem = m0 - img * a.howo;
                const int oh = rem / a.wo;
                const int ow = rem - oh * a.wo;
                const int corner_w = ow * a.stride_w - a.pad_w;
                const int corner_h = oh * a.stride_h - a.pad_h;
                // SWAP: the second 128-pixel box of the tile (may lie past the last
                // image: TMA then reads zeros).
                const int m1 = m0 + C::BM;
                const int img1 = m1 / a.howo;
                const int rem1 = m1 - img1 * a.howo;
                const int oh1 = rem1 / a.wo;
                const int ow1 = rem1 - oh1 * a.wo;
                const int corner_w1 = ow1 * a.stride_w - a.pad_w;
                const int corner_h1 = oh1 * a.stride_h - a.pad_h;
                // K step k reads filter tap k % taps of channel chunk k / taps: the taps run
                // fastest, so a tile's first steps read one chunk of its input rows, not all
                // of them (from a cold L2 the first stages arrive sooner; the deep 3x3 layer
                // measured 0.25 us faster than with the channel chunk fastest).
                const int taps = a.k_iters / a.c_chunks;
                int cc = u.kb / taps;
                int s = (u.kb - cc * taps) % a.s;
                int r = (u.kb - cc * taps) / a.s;
                bool ok = true;
                for (int it = u.kb; it < u.ke; ++it) {
                    const uint32_t e_bar = dev::smem_u32(&empty[stage]);
                    if (!dev::mbar_wait_bounded(e_bar, phase ^ 1u, abort_flag, a.wait_ns)) {
                        if (!*abort_flag) record_error(kErrTimeoutProducer, abort_flag);
                        ok = false;
                        break;
                    }
                    const uint32_t f_bar = dev::smem_u32(&full[stage]);
                    if constexpr (PAIR) {
                        // Both CTAs' bytes complete on the even CTA's full barrier.
                        const uint32_t f0 = full0 + (uint32_t)(stage * 8);
                        if (loads_w) {
                            if (rank == 0) dev::mbar_arrive_expect_tx(f_bar, 2 * C::B_BYTES);
                            dev::tma_load_3d_pair(dev::smem_u32(sm_b + stage * C::B_STRIDE), &tm_w, f0, cc * BK,
                                                  r * a.s + s, n0 + rank * (BN / 2));
                        } else {
                            if (rank == 0) dev::mbar_arrive_expect_tx(f_bar, 2 * C::A_BYTES);
                            dev::tma_load_im2col_4d_pair(dev::smem_u32(sm_a + stage * C::A_STRIDE), &tm_x, f0,
                                                         cc * BK, corner_w, corner_h, img, (uint16_t)s,
                                                         (uint16_t)r);
                        }
                    } else if constexpr (SWAP) {
                        if (loads_w) {
                            dev::mbar_arrive_expect_tx(f_bar, C::A_BYTES);
                            dev::tma_load_3d(dev::smem_u32(sm_a + stage * C::A_STRIDE), &tm_w, f_bar,
                                             cc * BK, r * a.s + s, n0);
                        } else {
                            dev::mbar_arrive_expect_tx(f_bar, (two_boxes ? 2 : 1) * C::BM * BK * 2);
                            const uint32_t bdst = dev::smem_u32(sm_b + stage * C::B_STRIDE);
                            dev::tma_load_im2col_4d(bdst, &tm_x, f_bar, cc * BK, corner_w, corner_h, img,
                                                    (uint16_t)s, (uint16_t)r);
                            if (two_boxes)
                                dev::tma_load_im2col_4d(bdst + C::BM * BK * 2, &tm_x, f_bar, cc * BK, corner_w1,
                                                        corner_h1, img1, (uint16_t)s, (uint16_t)r);
                        }
                    } else {
                        if (loads_w) {
                            dev::mbar_arrive_expect_tx(f_bar, C::B_BYTES);
                            dev::tma_load_3d(dev::smem_u32(sm_b + stage * C::B_STRIDE), &tm_w, f_bar,
                                             cc * BK, r * a.s + s, n0);
                        } else {
                            dev::mbar_arrive_expect_tx(f_bar, C::A_BYTES);
                            dev::tma_load_im2col_4d(dev::smem_u32(sm_a + stage * C::A_STRIDE), &tm_x, f_bar,
                                                    cc * BK, corner_w, corner_h, img, (uint16_t)s,
                                                    (uint16_t)r);
                        }
                    }
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++s == a.s) {
                        s = 0;
                        if (++r * a.s == taps) {
                            r = 0;
                            ++cc;
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // Every load issued must land before the CTA may exit.  The odd CTA of a
            // pair cannot see the full barrier its loads complete on; its loads have
            // landed once the MMAs that read them released the stage.
            // After one drain wait has run out (2 s), the copies issued before it have long
            // landed: the remaining stages are not waited for again.
            bool drain_ok = true;
            for (int i = 0; i < STAGES && drain_ok; ++i) {
                if ((issued >> i) & 1u) {
                    const uint32_t bar = (PAIR && rank != 0) ? dev::smem_u32(&empty[i]) : dev::smem_u32(&full[i]);
                    if (!dev::mbar_wait_bounded(bar, (issued_parity >> i) & 1u, nullptr, kWaitTimeoutNs)) {
                        record_error(kErrTimeoutDrain, abort_flag);
                        drain_ok = false;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = dev::idesc_bf16_f32(PAIR ? 2 * C::BM : C::BM, BN);
            // Descriptors are built once; per stage and per K step only the start
            // address field (16-byte units, low bits) advances.  The single issuing
            // thread must spend almost nothing per MMA or it, not the tensor core,
            // sets the pace.
            const uint64_t desc_a0 = dev::smem_desc_kmajor(dev::smem_u32(sm_a), C::ROW_A);
            const uint64_t desc_b0 = dev::smem_desc_kmajor(dev::smem_u32(sm_b), C::ROW_A);
            int stage = 0;
            uint32_t phase = 0;
            int lt = 0;
            bool ok = true;
            WorkIter wi(a, vb, vg);
            WorkUnit u;
            for (; ok && wi.next(a, u); ++lt) {
                const int buf = lt & 1;
                const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
                if (!dev::mbar_wait_bounded(dev::smem_u32(&tempty[buf]), tparity ^ 1u, abort_flag,
                                            a.wait_ns)) {
                    if (!*abort_flag) record_error(kErrTimeoutMma, abort_flag);
                    break;
                }
                dev::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
                // Balanced channel-major units: the MMA's N is the unit's pixel count
                // (rounded up to 16; the rows past it were loaded as zeros or neighbours
                // and are never stored).
                const uint32_t idesc_u =
                    (SWAP && a.balanced) ? dev::idesc_bf16_f32(C::BM, (u.np + 15) & ~15) : idesc;
                for (int it = u.kb; it < u.ke; ++it) {
                    if (!dev::mbar_wait_bounded(dev::smem_u32(&full[stage]), phase, abort_flag,
                                                a.wait_ns)) {
                        if (!*abort_flag) record_error(kErrTimeoutMma, abort_flag);
                        ok = false;
                        break;
                    }
                    dev::tc_fence_after_sync();
                    const uint64_t da = desc_a0 + (uint64_t)(stage * (C::A_STRIDE >> 4));
                    const uint64_t db = desc_b0 + (uint64_t)(stage * (C::B_STRIDE >> 4));
                    dev::tc_mma_bf16<CG>(d_tmem, da, db, idesc_u, it != u.kb ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < BK / 16; ++kk)
                        dev::tc_mma_bf16<CG>(d_tmem, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), idesc_u,
                                             1u);
                    if constexpr (PAIR)
                        dev::tc_commit_multicast<CG>(dev::smem_u32(&empty[stage]), (uint16_t)0x3);
                    else
                        dev::tc_commit<CG>(dev::smem_u32(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    dev::tc_commit_multicast<CG>(dev::smem_u32(&tfull[buf]), (uint16_t)0x3);
                else
                    dev::tc_commit<CG>(dev::smem_u32(&tfull[buf]));
            }
            // The helpers' one barrier: it completes once, when every MMA above has.
            if constexpr (HELP) dev::tc_commit_multicast<CG>(dev::smem_u32(lastfull), (uint16_t)0x3);
            // All MMAs issued by this thread must finish before TMEM is freed.
            dev::tc_commit<CG>(dev::smem_u32(drain));
            if (!dev::mbar_wait_bounded(dev::smem_u32(drain), 0, nullptr, kWaitTimeoutNs))
                record_error(kErrTimeoutDrain, abort_flag);
        }
        __syncwarp();
    }
    if ((warp >= 4 && warp - 4 < C::EPI_WARPS) || (HELP && warp < 4)) {
        // ------------------------------------------------------------ epilogue
        constexpr int EC = C::EC;
        constexpr int ROW_Y = EC * 2;
        const int ew = warp & 3;          // this warp may access TMEM lanes [32*ew, 32*ew+32)
        const bool helper = warp < 4;     // a loading or issuing warp: the last unit only
        const int ep = helper ? C::EPI_WARPS + warp : warp - 4;  // epilogue warp index
        // This warp's chunks of a pixel-major tile: `own` chunks from column col_base (set per
        // unit where the last unit is split four ways).
        int c_lo = (ep >> 2) * C::NCH / C::WPQ;
        int own = ((ep >> 2) + 1) * C::NCH / C::WPQ - c_lo;
        int col_base = c_lo * EC;
        // A helper stages its stores in the operand ring, idle once the last unit's MMAs are done.
        uint8_t *my_stg = helper ? sm_a + warp * 2 * C::STG_BYTES : sm_stg + ep * 2 * C::STG_BYTES;
        int sbuf = 0;
        int lt = 0;
        // Residual epilogue: the residual's tile for a chunk is loaded by TMA into the
        // staging buffer the chunk's output will be stored from (the same box of the
        // same-shaped tensor), while the chunk's accumulator is read and activated.
        uint32_t r_phase = 0;    // per staging buffer: parity of its load barrier's next phase
        uint32_t r_pending = 0;  // per staging buffer: a load issued and not yet waited for
        auto residual_load = [&](int c0, int c1) {
            if (lane == 0) {
                dev::bulk_wait_group_read<1>();  // the buffer's previous store has read it
                const uint32_t bar = dev::smem_u32(&rbar[2 * ep + sbuf]);
                dev::mbar_arrive_expect_tx(bar, C::STG_BYTES);
                dev::tma_load_2d(dev::smem_u32(my_stg + sbuf * C::STG_BYTES), &tm_r, bar, c0, c1);
            }
            r_pending |= 1u << sbuf;
            __syncwarp();
        };
        auto residual_wait = [&]() {
            const uint32_t bar = dev::smem_u32(&rbar[2 * ep + sbuf]);
            const bool ok = dev::mbar_wait_bounded(bar, (r_phase >> sbuf) & 1u, abort_flag, a.wait_ns);
            r_phase ^= 1u << sbuf;
            r_pending &= ~(1u << sbuf);
            if (!__all_sync(0xffffffffu, ok) && lane == 0 && !*abort_flag)
                record_error(kErrTimeoutEpilogue, abort_flag);
        };
        const int row = ew * 32 + lane;  // this thread's row of the tile (TMEM lane)
        WorkIter wi(a, vb, vg);
        WorkUnit u;
        // SWAP: a unit's channel tile, first pixel and count of EC-pixel chunks.  The
        // warps of a lane quarter take the chunks in turn.
        const int half = ep >> 2;
        auto swap_geometry = [&](const WorkUnit &q, int &nt, int &p0, int &nchunks) {
            if (a.balanced) {
                nt = q.tile;
                p0 = q.p0;
                nchunks = (q.np + EC - 1) / EC;
            } else {
                const int pt = q.tile / a.n_tiles;
                nt = q.tile - pt * a.n_tiles;
                p0 = pt * BN;
                nchunks = BN / EC;
            }
        };
        // Residual epilogue: bring a unit's residual rows (this warp's part) into L2
        // while its K loop runs, so that the epilogue's loads of them hit L2.
        auto prefetch_residual = [&](const WorkUnit &q) {
            if constexpr (RES) {
                if constexpr (SWAP) {
                    int nt, p0, nchunks;
                    swap_geometry(q, nt, p0, nchunks);
                    const int chw = nt * C::BM + ew * 32;
                    if (chw < a.c_out) {
                        for (int j = half; j < nchunks; j += C::WPQ) {
                            const int px = p0 + j * EC + lane;  // EC == 32 on this path
                            if (px < a.m) prefetch_l2(a.residual + (size_t)px * a.c_out + chw);
                        }
                    }
                } else {
                    const int mu = q.tile / a.n_tiles;
                    const int mt = PAIR ? 2 * mu + rank : mu;
                    const int c0 = (q.tile - mu * a.n_tiles) * BN + col_base;
                    const int px = mt * C::BM + ew * 32 + lane;
                    if (px < a.m && c0 < a.c_out) {
                        const int bytes = 2 * (a.c_out - c0 < own * EC ? a.c_out - c0 : own * EC);
                        const char *rp = reinterpret_cast<const char *>(a.residual + (size_t)px * a.c_out + c0);
                        for (int b = 0; b < bytes; b += 128) prefetch_l2(rp + b);
                    }
                }
            }
        };
        if constexpr (RES) {
            WorkIter first = wi;
            WorkUnit q;
            if (first.next(a, q)) prefetch_residual(q);
        }
        for (; wi.next(a, u); ++lt) {
            const int buf = lt & 1;
            const uint32_t tparity = (uint32_t)(lt >> 1) & 1u;
            if constexpr (HELP) {
                // The worker's last unit: four warps per lane quarter, two chunks each.
                WorkIter nx = wi;
                WorkUnit q;
                const bool last = !nx.next(a, q);
                if (helper && !last) continue;
                const int parts = last ? C::WPQ + 1 : C::WPQ;
                c_lo = (ep >> 2) * C::NCH / parts;
                own = ((ep >> 2) + 1) * C::NCH / parts - c_lo;
                col_base = c_lo * EC;
            }
            // Stream-K, pixel-major tiles: the two pieces of a split tile (the head of one
            // worker's range and the tail of the next one's) meet in the slot of that worker
            // boundary; a pair keeps one partial tile per M half.  Each worker runs its head
            // piece first, so the head piece publishes its fp32 partial sums and the tail
            // piece, which its worker runs later, adds them and finishes the tile.  A sum of
            // two fp32 values does not depend on their order: the result is deterministic.
            const bool split = !SWAP && a.stream_k && (u.kb > 0 || u.ke < a.k_iters);
            const bool publish = split && u.kb == 0;
            const bool combine = split && u.kb > 0;
            const int slot = (u.kb > 0 ? vb - 1 : vb) * (PAIR ? 2 : 1) + rank;
            float4 *part = a.stream_k ? reinterpret_cast<float4 *>(a.partial) + (size_t)slot * (32 * BN)
                                      : nullptr;
            // The unit's per-channel scale and bias, read while its K loop still runs: the
            // first touch of these lines otherwise costs an L2 round trip inside the epilogue.
            float swap_hs = 0.f, swap_hb = 0.f;  // channel-major tiles: this thread's channel
            if constexpr (SWAP) {
                const int nt = a.balanced ? u.tile : u.tile - (u.tile / a.n_tiles) * a.n_tiles;
                const int ch = nt * C::BM + ew * 32 + lane;
                swap_hs = ch < a.c_out ? 0.5f * __ldg(a.scale + ch) : 0.f;
                swap_hb = ch < a.c_out ? 0.5f * __ldg(a.bias + ch) : 0.f;
            } else {
                // One prefetch per 16 channels (64 bytes) of each array, so that every 128-byte
                // line the warp's columns touch is covered whatever the arrays' alignment.
                const int c0 = (u.tile - (u.tile / a.n_tiles) * a.n_tiles) * BN + col_base;
                constexpr int NP = (C::MAX_OWN * EC + 15) / 16;
                static_assert(2 * NP <= 32, "one lane per prefetch");
                if (lane < 2 * NP) {
                    const int c = c0 + (lane % NP) * 16;
                    if (c < a.c_out && c < c0 + own * EC) prefetch_l1(lane < NP ? a.scale + c : a.bias + c);
                }
            }
            // Stream-K flags: one per (lane quarter, 32-column chunk) of the tile, so that the two
            // pieces of a tile may split its columns among their warps differently.  A combining
            // warp reads its chunks' flags now, while it waits for the accumulator anyway: they
            // are nearly always up by then, and the loads' L2 round trip (~1 us at the end of the
            // kernel) stays out of the epilogue.
            int *const fl = split ? a.flags + slot * kTcFlagsPerSlot + ew * C::NCH + c_lo : nullptr;
            uint32_t seen = 0;  // combine: this warp's chunks whose flag is already up
            if (combine) seen = __ballot_sync(0xffffffffu, lane < own && ld_acquire_gpu(fl + lane) != 0);
            // A helper comes to its wait after an unknown number of the buffer's earlier phases
            // (a parity wait only tells the last two apart), so it waits on a barrier of its own
            // that completes once, after the worker's last MMA.
            const uint32_t fbar = helper ? dev::smem_u32(lastfull) : dev::smem_u32(&tfull[buf]);
            const uint32_t fpar = helper ? 0u : tparity;
            int ok = 1;
            if (lane == 0) ok = dev::mbar_wait_bounded(fbar, fpar, abort_flag, a.wait_ns) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0 && !*abort_flag) record_error(kErrTimeoutEpilogue, abort_flag);
                break;
            }
            dev::tc_fence_after_sync();
            if constexpr (RES) {
                WorkIter after = wi;  // already past u
                WorkUnit q;
                if (after.next(a, q)) prefetch_residual(q);
            }
            if constexpr (SWAP) {
                // TMEM lane = output channel, column = pixel.  Each thread owns one
                // channel, so BN scale/bias are per-thread constants; the tile is
                // transposed to NHWC through shared memory, 32 pixels x 32 channels
                // per TMA store.
                int nt, p0, nchunks;
                swap_geometry(u, nt, p0, nchunks);
                const int ch_w0 = nt * C::BM + ew * 32;  // warp's first channel
                const float hs = swap_hs, hb = swap_hb;
                const uint32_t t_lane = tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(buf * BN);
                if (half >= nchunks) {
                    // A unit narrower than two chunks leaves this warp nothing to read.
                    dev::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                }
#pragma unroll 1
                for (int j = half; j < nchunks; j += C::WPQ) {
                    // A chunk wholly past the last pixel or channel is skipped (no staging write
                    // without its store: the wait before each write counts one store per chunk).
                    if (p0 + j * EC >= a.m || ch_w0 >= a.c_out) {
                        if (j + C::WPQ >= nchunks) {
                            dev::tc_fence_before_sync();
                            __syncwarp();
                            if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                        }
                        continue;
                    }
                    if constexpr (RES) residual_load(ch_w0, p0 + j * EC);
                    uint32_t v[EC];
#pragma unroll
                    for (int q = 0; q < EC / 16; ++q)
                        dev::tmem_ld_32x32b_x16(t_lane + (uint32_t)(j * EC + q * 16), v + q * 16);
                    dev::tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < EC / 16; ++q) dev::reg_fence16(v + q * 16);
                    if (j + C::WPQ >= nchunks) {
                        // This warp's last chunk is in registers: release the accumulator.
                        dev::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                    }
                    if (lane == 0) dev::bulk_wait_group_read<1>();
                    __syncwarp();
                    // Staging rows: row pp holds pixel pp's 32 channels (2 bytes each, or 1 for fp8).
                    const uint32_t sb = dev::smem_u32(my_stg + sbuf * C::STG_BYTES);
                    const int px0 = p0 + j * EC;
                    with_epi_mode<EPI>(emode, [&](auto mode_c) {
                        constexpr int md = decltype(mode_c)::value;
                        if constexpr (FP8) {
#pragma unroll
                            for (int pp = 0; pp < EC; ++pp)  // row pp: 32 channels, one byte per lane
                                dev::sts_u8(sb + (uint32_t)(pp * 32 + lane),
                                            dev::to_e4m3(dev::epilogue_from_half(__uint_as_float(v[pp]), hs, hb, md)));
                        } else if constexpr (RES) {
                            // The residual tile is in the staging buffer (row pp: the pixel's 32
                            // channels); each lane adds its channel's column in place.
                            float f[EC];
#pragma unroll
                            for (int pp = 0; pp < EC; ++pp)
                                f[pp] = dev::epilogue_from_half(__uint_as_float(v[pp]), hs, hb, md);
                            residual_wait();
#pragma unroll
                            for (int pp = 0; pp < EC; ++pp) {
                                const uint32_t at = sb + (uint32_t)((pp * 32 + lane) * 2);
                                dev::sts_u16(at, __bfloat16_as_ushort(__float2bfloat16_rn(
                                                     f[pp] + dev::bf16_bits_to_float(dev::lds_u16(at)))));
                            }
                        } else {
#pragma unroll
                            for (int pp = 0; pp < EC; ++pp)  // row pp: 32 channels, one per lane
                                dev::sts_u16(sb + (uint32_t)((pp * 32 + lane) * 2),
                                             __bfloat16_as_ushort(__float2bfloat16_rn(
                                                 dev::epilogue_from_half(__uint_as_float(v[pp]), hs, hb, md))));
                        }
                    });
                    dev::fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {  // a live chunk: TMA clips the pixels past m
                        dev::tma_store_2d(&tm_y, sb, ch_w0, px0);
                        dev::bulk_commit_group();
                    }
                    sbuf ^= 1;
                }
                continue;
            }
            const int m_unit = u.tile / a.n_tiles;
            const int m_tile = PAIR ? 2 * m_unit + rank : m_unit;
            const int n0 = (u.tile - m_unit * a.n_tiles) * BN;
            const int row0 = m_tile * C::BM + ew * 32;  // first output pixel of this warp
            bool timed_out = false;
            const uint32_t t_lane =
                tmem_base + ((uint32_t)(ew * 32) << 16) + (uint32_t)(buf * BN + col_base);
#pragma unroll 1
            for (int j = 0; j < own; ++j) {
                // A chunk wholly past the last output channel or pixel is skipped: nothing of it
                // is stored (nor published), and it must not touch a staging buffer either, since
                // the wait before each staging write counts one store per staged chunk.
                if (row0 >= a.m || n0 + col_base + j * EC >= a.c_out) {
                    if (j == own - 1 && !helper) {
                        dev::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if (PAIR && rank != 0)
                                dev::mbar_arrive_cluster(tempty0 + (uint32_t)(buf * 8));
                            else
                                dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                        }
                    }
                    continue;
                }
                if constexpr (RES)
                    if (!publish) residual_load(n0 + col_base + j * EC, row0);
                uint32_t v[EC];
#pragma unroll
                for (int q = 0; q < EC / 16; ++q)
                    dev::tmem_ld_32x32b_x16(t_lane + (uint32_t)(j * EC + q * 16), v + q * 16);
                dev::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < EC / 16; ++q) dev::reg_fence16(v + q * 16);
                if (j == own - 1 && !helper) {
                    // The accumulator is in registers: hand the TMEM buffer back to the MMA warp
                    // (the helpers read the last unit, which the MMA warp does not wait for).
                    dev::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR && rank != 0)
                            dev::mbar_arrive_cluster(tempty0 + (uint32_t)(buf * 8));
                        else
                            dev::mbar_arrive(dev::smem_u32(&tempty[buf]));
                    }
                }
                if (publish) {
                    // Column-group-major, row-minor: a warp writes 512 contiguous bytes per store.
#pragma unroll
                    for (int q = 0; q < EC / 4; ++q)
                        __stcg(part + (size_t)((col_base + j * EC) / 4 + q) * C::BM + row,
                               make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                           __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
                    // The warp barrier orders every lane's stores of the chunk before lane 0's
                    // release store of its flag, which makes them visible with it GPU-wide.  (A
                    // sequentially consistent GPU-scope fence on either side of this handoff
                    // cost ~2 us per combined tile, on the kernel's critical path.)
                    __syncwarp();
                    if (lane == 0) st_release_gpu(fl + j, 1);
                    continue;
                }
                if (combine) {
                    if (!((seen >> j) & 1u)) {
                        int got = 1;
                        if (lane == 0) got = wait_flag_bounded(fl + j, abort_flag, a.wait_ns) ? 1 : 0;
                        if (!__shfl_sync(0xffffffffu, got, 0)) {
                            if (lane == 0 && !*abort_flag) record_error(kErrTimeoutEpilogue, abort_flag);
                            timed_out = true;
                            break;
                        }
                    }
                    // The flag was seen by an acquire load of one lane; the warp barrier orders
                    // that before every lane's loads of the partial sums.
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < EC / 4; ++q) {
                        const float4 p4 = __ldcg(part + (size_t)((col_base + j * EC) / 4 + q) * C::BM + row);
                        v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) + p4.x);
                        v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + p4.y);
                        v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + p4.z);
                        v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + p4.w);
                    }
                    // The chunk's partial sums are read: its flag goes back down for the next
                    // launch (nothing else in this one waits for it).
                    if (lane == 0) st_release_gpu(fl + j, 0);
                }
                const int ch0 = n0 + col_base + j * EC;
                uint32_t packed[EC / 2];
                uint32_t q8[FP8 ? EC / 4 : 1];
                // The activation is a compile-time constant in each arm: the fused layer's
                // instantiation has SiLU alone; the others pick the arm once per chunk.
                auto activate = [&](auto mode_c) {
                    constexpr int md = decltype(mode_c)::value;
                    if constexpr (FP8) {
                        // fp8 output: each value rounded once, from fp32 straight to e4m3.
#pragma unroll
                        for (int i = 0; i < EC; i += 4) {
                            float f[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int c = ch0 + i + e;
                                f[e] = c < a.c_out ? dev::epilogue_value(__uint_as_float(v[i + e]), __ldg(a.scale + c),
                                                                         __ldg(a.bias + c), md)
                                                   : 0.f;
                            }
                            q8[i / 4] = dev::pack_e4m3x4(f[0], f[1], f[2], f[3]);
                        }
                    } else if constexpr (RES) {
                        // With a residual: its tile is in the staging buffer, swizzled like the
                        // output tile; this lane's row, 8 channels per 16-byte piece.
                        float f[EC];
                        if (ch0 + EC <= a.c_out) {
#pragma unroll
                            for (int i = 0; i < EC; i += 4) {
                                const float4 sc = __ldg(reinterpret_cast<const float4 *>(a.scale + ch0 + i));
                                const float4 bi = __ldg(reinterpret_cast<const float4 *>(a.bias + ch0 + i));
                                f[i] = dev::epilogue_value(__uint_as_float(v[i]), sc.x, bi.x, md);
                                f[i + 1] = dev::epilogue_value(__uint_as_float(v[i + 1]), sc.y, bi.y, md);
                                f[i + 2] = dev::epilogue_value(__uint_as_float(v[i + 2]), sc.z, bi.z, md);
                                f[i + 3] = dev::epilogue_value(__uint_as_float(v[i + 3]), sc.w, bi.w, md);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < EC; ++i) {
                                const int c = ch0 + i;
                                f[i] = c < a.c_out ? dev::epilogue_value(__uint_as_float(v[i]), __ldg(a.scale + c),
                                                                         __ldg(a.bias + c), md)
                                                   : 0.f;
                            }
                        }
                        residual_wait();
                        const uint32_t rb = dev::smem_u32(my_stg + sbuf * C::STG_BYTES);
#pragma unroll
                        for (int q = 0; q < ROW_Y / 16; ++q) {
                            const uint4 r4 = dev::lds_v4(rb + swizzle_offset<ROW_Y>((uint32_t)(lane * ROW_Y + q * 16)));
                            const uint32_t rw[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                packed[4 * q + e] = dev::pack_bf16x2(f[8 * q + 2 * e] + __uint_as_float(rw[e] << 16),
                                                                     f[8 * q + 2 * e + 1] +
                                                                         __uint_as_float(rw[e] & 0xffff0000u));
                        }
                    } else if (ch0 + EC <= a.c_out) {
#pragma unroll
                        for (int i = 0; i < EC; i += 4) {
                            const float4 sc = __ldg(reinterpret_cast<const float4 *>(a.scale + ch0 + i));
                            const float4 bi = __ldg(reinterpret_cast<const float4 *>(a.bias + ch0 + i));
                            packed[i / 2] = dev::pack_bf16x2(
                                dev::epilogue_value(__uint_as_float(v[i]), sc.x, bi.x, md),
                                dev::epilogue_value(__uint_as_float(v[i + 1]), sc.y, bi.y, md));
                            packed[i / 2 + 1] =
                                dev::pack_bf16x2(dev::epilogue_value(__uint_as_float(v[i + 2]), sc.z, bi.z, md),
                                                 dev::epilogue_value(__uint_as_float(v[i + 3]), sc.w, bi.w, md));
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < EC; i += 2) {
                            const int c0 = ch0 + i, c1 = ch0 + i + 1;
                            const float s0 = c0 < a.c_out ? __ldg(a.scale + c0) : 0.f;
                            const float b0 = c0 < a.c_out ? __ldg(a.bias + c0) : 0.f;
                            const float s1 = c1 < a.c_out ? __ldg(a.scale + c1) : 0.f;
                            const float b1 = c1 < a.c_out ? __ldg(a.bias + c1) : 0.f;
                            packed[i / 2] = dev::pack_bf16x2(dev::epilogue_value(__uint_as_float(v[i]), s0, b0, md),
                                                             dev::epilogue_value(__uint_as_float(v[i + 1]), s1, b1, md));
                        }
                    }
                };
                with_epi_mode<EPI>(emode, activate);
                // Stage the warp's 32 rows x EC channels, then one TMA store.
                if (lane == 0) dev::bulk_wait_group_read<1>();
                __syncwarp();
                const uint32_t sb = dev::smem_u32(my_stg + sbuf * C::STG_BYTES);
                if constexpr (FP8) {
                    // One byte per value: rows of EC bytes (32: 32-byte swizzle; 16: none).
#pragma unroll
                    for (int q = 0; q < EC / 16; ++q) {
                        const uint32_t raw = (uint32_t)(lane * EC + q * 16);
                        const uint32_t off = EC == 32 ? swizzle_offset<32>(raw) : raw;
                        dev::sts_v4(sb + off, q8[4 * q], q8[4 * q + 1], q8[4 * q + 2], q8[4 * q + 3]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < ROW_Y / 16; ++q) {
                        const uint32_t off = swizzle_offset<ROW_Y>((uint32_t)(lane * ROW_Y + q * 16));
                        dev::sts_v4(sb + off, packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                    }
                }
                dev::fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {  // a live chunk: TMA clips the channels past c_out and rows past m
                    dev::tma_store_2d(&tm_y, sb, ch0, row0);
                    dev::bulk_commit_group();
                }
                sbuf ^= 1;
            }
            if (timed_out) break;
        }
        if constexpr (RES) {
            // Only after a wait ran out can a load still be in flight: wait for it once more
            // (bounded) before the CTA's shared memory is given up.
            for (int b = 0; b < 2; ++b)
                if ((r_pending >> b) & 1u) {
                    const bool ok = dev::mbar_wait_bounded(dev::smem_u32(&rbar[2 * ep + b]), (r_phase >> b) & 1u,
                                                           nullptr, kWaitTimeoutNs);
                    if (!ok && lane == 0) record_error(kErrTimeoutDrain, abort_flag);
                }
        }
        if (lane == 0) dev::bulk_wait_group<0>();
        __syncwarp();
    }

    dev::tc_fence_before_sync();
    __syncthreads();
    if constexpr (PAIR) dev::cluster_sync();  // no CTA leaves while its peer may still write to it
    if (warp == 1) {
        dev::tc_fence_after_sync();
        dev::tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

cudaError_t load_encoders()
{
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q1, q2;
        void *f1 = nullptr, *f2 = nullptr;
        cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000,
                                                          cudaEnableDefault, &q1);
        cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &f2, 12000,
                                                          cudaEnableDefault, &q2);
        if (e1 != cudaSuccess || e2 != cudaSuccess || q1 != cudaDriverEntryPointSuccess ||
            q2 != cudaDriverEntryPointSuccess || !f1 || !f2) {
            g_encode_status = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : cudaErrorNotSupported);
            return;
        }
        g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
        g_encode_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(f2);
    });
    return g_encode_status;
}

CUtensorMapSwizzle swizzle_for_row_bytes(int row_bytes)
{
    return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                            : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

struct TcMaps {
    CUtensorMap x, w, y;
    CUtensorMap r;  // the residual, laid out and boxed like y (a copy of y's map when there is none)
};

// A bf16 NHWC tensor shaped like y ([m][c_out]) at `base`, viewed as (C_out, M) with the
// epilogue's store box: (EC, 32) with the EC-channel swizzle, or for swap AB (32, EC),
// unswizzled 64-byte rows.  y itself, and the residual the epilogue adds, which it
// loads tile by tile into the same staging buffer that y's tile is stored from.
static cudaError_t encode_bf16_like_y(const ConvProblem &p, int block_n, bool swap, const void *base,
                                      CUtensorMap *out)
{
    int split = 1, ec = 16;
    tc_epilogue_geometry(block_n, &split, &ec);
    cuuint64_t dims[2] = {(cuuint64_t)p.c_out, (cuuint64_t)p.m};
    cuuint64_t strides[1] = {(cuuint64_t)p.c_out * 2};
    cuuint32_t box[2] = {(cuuint32_t)(swap ? 32 : ec), (cuuint32_t)(swap ? ec : 32)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swap ? CU_TENSOR_MAP_SWIZZLE_NONE : swizzle_for_row_bytes(ec * 2),
                                CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t tc_encode_x_im2col(const ConvProblem &p, int block_k, int box_pixels, CUtensorMap *out)
{
    cudaError_t st = load_encoders();
    if (st != cudaSuccess) return st;
    // x: im2col view over (C, W, H, N).  The bounding box of window corners is
    // [-pad, dim - 1 + pad - (filter - 1)] along W and H, traversed with the
    // convolution stride, so a box of `box_pixels` pixels walks output pixels in
    // (img, oh, ow) order, crossing rows and images.
    cuuint64_t dims[4] = {(cuuint64_t)p.c, (cuuint64_t)p.w_in, (cuuint64_t)p.h, (cuuint64_t)p.n};
    cuuint64_t strides[3] = {(cuuint64_t)p.c * 2, (cuuint64_t)p.w_in * p.c * 2, (cuuint64_t)p.h * p.w_in * p.c * 2};
    int lower[2] = {-p.pad_w, -p.pad_h};
    int upper[2] = {p.pad_w - (p.s - 1), p.pad_h - (p.r - 1)};
    cuuint32_t estr[4] = {1, (cuuint32_t)p.stride_w, (cuuint32_t)p.stride_h, 1};
    CUresult r = g_encode_im2col(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.x), dims, strides,
                                 lower, upper, (cuuint32_t)block_k, (cuuint32_t)box_pixels, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(block_k * 2),
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_encode_x_rows(const ConvProblem &p, int block_k, int rows, CUtensorMap *out)
{
    cudaError_t st = load_encoders();
    if (st != cudaSuccess) return st;
    // x viewed as (stride*C, W/stride, H, N): input pixel stride*j + e is element e of view
    // pixel j.  Box: block_k channels of wo view pixels over `rows` input rows taken every
    // stride-th row (the rows one filter tap of `rows` output rows reads).
    const int sd = p.stride_w;
    cuuint64_t dims[4] = {(cuuint64_t)sd * p.c, (cuuint64_t)(p.w_in / sd), (cuuint64_t)p.h, (cuuint64_t)p.n};
    cuuint64_t strides[3] = {(cuuint64_t)sd * p.c * 2, (cuuint64_t)p.w_in * p.c * 2, (cuuint64_t)p.h * p.w_in * p.c * 2};
    cuuint32_t box[4] = {(cuuint32_t)block_k, (cuuint32_t)p.wo, (cuuint32_t)(p.stride_h * (rows - 1) + 1), 1};
    cuuint32_t estr[4] = {1, 1, (cuuint32_t)p.stride_h, 1};
    CUresult r = g_encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.x), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(block_k * 2),
                                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_encode_x_matrix(const ConvProblem &p, int block_k, int box_rows, CUtensorMap *out)
{
    cudaError_t st = load_encoders();
    if (st != cudaSuccess) return st;
    cuuint64_t dims[2] = {(cuuint64_t)p.c, (cuuint64_t)p.m};
    cuuint64_t strides[1] = {(cuuint64_t)p.c * 2};
    cuuint32_t box[2] = {(cuuint32_t)block_k, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.x), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(block_k * 2),
                                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_encode_w_tile(const ConvProblem &p, int block_k, int rows, CUtensorMap *out)
{
    cudaError_t st = load_encoders();
    if (st != cudaSuccess) return st;
    // W: (C, R*S, C_out), box (BK, 1, rows): one filter tap's BK channels of `rows` output channels.
    cuuint64_t dims[3] = {(cuuint64_t)p.c, (cuuint64_t)p.r * p.s, (cuuint64_t)p.c_out};
    cuuint64_t strides[2] = {(cuuint64_t)p.c * 2, (cuuint64_t)p.r * p.s * p.c * 2};
    cuuint32_t box[3] = {(cuuint32_t)block_k, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.w), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for_row_bytes(block_k * 2),
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_encode_y_rows(const ConvProblem &p, const void *base, int box_c, int box_m, CUtensorMap *out)
{
    cudaError_t st = load_encoders();
    if (st != cudaSuccess) return st;
    // A tensor shaped like y, viewed as (C_out, M), unswizzled box (box_c, box_m); bf16, or
    // one byte per element for the fp8 output.
    cuuint64_t dims[2] = {(cuuint64_t)p.c_out, (cuuint64_t)p.m};
    cuuint64_t strides[1] = {(cuuint64_t)p.c_out * (p.out_fp8 ? 1 : 2)};
    cuuint32_t box[2] = {(cuuint32_t)box_c, (cuuint32_t)box_m};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(out, p.out_fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

cudaError_t encode_maps(const ConvProblem &p, int block_n, int block_k, bool swap, bool pair, TcMaps *maps)
{
    cudaError_t st = tc_encode_x_im2col(p, block_k, kTcBlockM, &maps->x);
    if (st != cudaSuccess) return st;
    // W rows of one load: the whole N tile, the 128-channel A tile when swapped, or half
    // the N tile per CTA of a 2-CTA pair.
    st = tc_encode_w_tile(p, block_k, swap ? kTcBlockM : (pair ? block_n / 2 : block_n), &maps->w);
    if (st != cudaSuccess) return st;
    // y: (C_out, M), box (EC, 32): one epilogue warp's rows, one column chunk.
    if (p.out_fp8) {
        // fp8 e4m3 output, one byte per element: rows of EC bytes (pixel-major), or for
        // swap AB rows of 32 one-byte channels, EC pixels (unswizzled).
        int split = 1, ec = 16;
        tc_epilogue_geometry(block_n, &split, &ec);
        cuuint64_t dims[2] = {(cuuint64_t)p.c_out, (cuuint64_t)p.m};
        cuuint64_t strides[1] = {(cuuint64_t)p.c_out};
        cuuint32_t box[2] = {(cuuint32_t)(swap ? 32 : ec), (cuuint32_t)(swap ? ec : 32)};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = g_encode_tiled(&maps->y, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, p.y, dims, strides, box, estr,
                                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                                    (!swap && ec == 32) ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        maps->r = maps->y;
        return cudaSuccess;
    }
    st = encode_bf16_like_y(p, block_n, swap, p.y, &maps->y);
    maps->r = maps->y;
    return st;
}

// Encoded tensor maps of recent calls, keyed by pointers, shape and tile.  Encoding
// is a driver call; layers called repeatedly on the same buffers reuse it.
struct MapKey {
    const void *x, *w, *y;
    int dims[11];
    int block_n, block_k, device, swap, pair, fp8;
    bool operator==(const MapKey &o) const
    {
        if (x != o.x || w != o.w || y != o.y || block_n != o.block_n || block_k != o.block_k ||
            device != o.device || swap != o.swap || pair != o.pair || fp8 != o.fp8)
            return false;
        for (int i = 0; i < 11; ++i)
            if (dims[i] != o.dims[i]) return false;
        return true;
    }
};

struct MapCache {
    static constexpr int kSlots = 64;
    std::mutex mu;
    MapKey keys[kSlots];
    TcMaps maps[kSlots];
    bool used[kSlots] = {};
    int next = 0;
};

MapCache g_map_cache;

cudaError_t cached_maps(const ConvProblem &p, int block_n, int block_k, bool swap, bool pair, TcMaps *out)
{
    MapKey k{};
    k.x = p.x;
    k.w = p.w;
    k.y = p.y;
    const int d[11] = {p.n, p.h, p.w_in, p.c, p.c_out, p.r, p.s, p.stride_h, p.stride_w, p.pad_h, p.pad_w};
    for (int i = 0; i < 11; ++i) k.dims[i] = d[i];
    k.block_n = block_n;
    k.block_k = block_k;
    k.swap = swap ? 1 : 0;
    k.pair = pair ? 1 : 0;
    k.fp8 = p.out_fp8;
    cudaError_t st = cudaGetDevice(&k.device);
    if (st != cudaSuccess) return st;
    {
        std::lock_guard<std::mutex> lock(g_map_cache.mu);
        for (int i = 0; i < MapCache::kSlots; ++i) {
            if (g_map_cache.used[i] && g_map_cache.keys[i] == k) {
                *out = g_map_cache.maps[i];
                return cudaSuccess;
            }
        }
    }
    st = encode_maps(p, block_n, block_k, swap, pair, out);
    if (st != cudaSuccess) return st;
    std::lock_guard<std::mutex> lock(g_map_cache.mu);
    const int slot = g_map_cache.next;
    g_map_cache.next = (slot + 1) % MapCache::kSlots;
    g_map_cache.keys[slot] = k;
    g_map_cache.maps[slot] = *out;
    g_map_cache.used[slot] = true;
    return cudaSuccess;
}

// Stream-K scratch, one buffer per (device, stream) so that calls on different
// streams never share it; grown on demand with cudaMalloc, ready flags zeroed
// when (re)allocated.  Kernels leave every flag at zero when they finish.
struct Workspace {
    int device;
    cudaStream_t stream;
    void *ptr;
    size_t bytes, flag_bytes;
};
std::mutex g_ws_mu;
Workspace g_ws[kWorkspaceStreams];
int g_ws_count = 0;

// The buffer is a zeroed flag region followed by the partial tiles.  Plans differ in
// how many flags they use; every plan's partial tiles start after the buffer's whole
// flag region (`*flag_region`), so that no plan's partial sums land where another
// plan's flags live.
cudaError_t stream_k_workspace(cudaStream_t stream, size_t partial_bytes, size_t flag_bytes, void **out,
                               size_t *flag_region)
{
    int device = 0;
    cudaError_t st = cudaGetDevice(&device);
    if (st != cudaSuccess) return st;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace *w = nullptr;
    for (int i = 0; i < g_ws_count; ++i)
        if (g_ws[i].device == device && g_ws[i].stream == stream) w = &g_ws[i];
    if (w && w->ptr && w->flag_bytes >= flag_bytes && w->bytes - w->flag_bytes >= partial_bytes) {
        *out = w->ptr;
        *flag_region = w->flag_bytes;
        return cudaSuccess;
    }
    if (w) {  // grow both parts, never shrink either
        flag_bytes = std::max(flag_bytes, w->flag_bytes);
        partial_bytes = std::max(partial_bytes, w->bytes - w->flag_bytes);
    }
    const size_t bytes = flag_bytes + partial_bytes;
    if (!w) {
        if (g_ws_count == kWorkspaceStreams) return cudaErrorMemoryAllocation;  // tc_workspace_reserve said no
        w = &g_ws[g_ws_count++];
        *w = Workspace{device, stream, nullptr, 0, 0};
    } else if (w->ptr) {
        st = cudaStreamSynchronize(stream);  // the old buffer may still be in use
        if (st != cudaSuccess) return st;
        cudaFree(w->ptr);
        w->ptr = nullptr;
        w->bytes = w->flag_bytes = 0;
    }
    void *ptr = nullptr;
    st = cudaMalloc(&ptr, bytes);
    if (st != cudaSuccess) return st;
    st = cudaMemsetAsync(ptr, 0, flag_bytes, stream);
    if (st != cudaSuccess) {
        cudaFree(ptr);
        return st;
    }
    w->ptr = ptr;
    w->bytes = bytes;
    w->flag_bytes = flag_bytes;
    *out = ptr;
    *flag_region = flag_bytes;
    return cudaSuccess;
}

template <int BN, int BK, bool SWAP, bool PAIR, int EPI>
cudaError_t launch_cfg(const ConvProblem &p, const TcPlan &plan, const TcMaps &maps, cudaStream_t stream,
                       void *caller_workspace)
{
    using C = TcCfg<BN, BK, PAIR ? BN / 2 : BN, PAIR>;
    auto kern = tc_conv_bn_silu_kernel<BN, BK, SWAP, PAIR, EPI>;
    // The shared-memory opt-in is per function and device: done once per device.
    static std::mutex attr_mu;
    static unsigned long long attr_done = 0;  // bit per device ordinal (< 64)
    int device = 0;
    cudaError_t st = cudaGetDevice(&device);
    if (st != cudaSuccess) return st;
    {
        std::lock_guard<std::mutex> lock(attr_mu);
        const unsigned long long bit = device < 64 ? (1ull << device) : 0ull;
        if (!(attr_done & bit) || bit == 0) {
            st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
            if (st != cudaSuccess) return st;
            attr_done |= bit;
        }
    }
    TcArgs a;
    a.scale = p.scale;
    a.bias = p.bias;
    a.c_out = p.c_out;
    a.m = (int)p.m;
    a.n_tiles = plan.n_tiles;
    a.tiles = plan.tiles;
    a.howo = p.ho * p.wo;
    a.wo = p.wo;
    a.stride_h = p.stride_h;
    a.stride_w = p.stride_w;
    a.pad_h = p.pad_h;
    a.pad_w = p.pad_w;
    a.s = p.s;
    a.c_chunks = plan.c_chunks;
    a.k_iters = plan.k_iters;
    a.epi_mode = p.epi_mode;
    a.residual = static_cast<const __nv_bfloat16 *>(p.residual);
    a.stream_k = plan.stream_k;
    a.wait_ns = p.wait_timeout_ns > 0 ? (unsigned long long)p.wait_timeout_ns : kWaitTimeoutNs;
    a.partial = nullptr;
    a.flags = nullptr;
    a.balanced = plan.swap_ab ? plan.balanced : 0;
    a.chunks_m = (int)((p.m + 31) / 32);
    if (plan.stream_k) {
        void *ws = caller_workspace;
        size_t flag_region = (size_t)plan.flag_bytes;  // a caller's buffer is laid out as the plan says
        if (ws == nullptr) {
            st = stream_k_workspace(stream, (size_t)(plan.workspace_bytes - plan.flag_bytes),
                                    (size_t)plan.flag_bytes, &ws, &flag_region);
            if (st != cudaSuccess) return st;
        }
        a.flags = static_cast<int *>(ws);
        a.partial = reinterpret_cast<float *>(static_cast<char *>(ws) + flag_region);
    }
    return launch_overlapped(kern, dim3((unsigned)plan.grid), dim3(C::THREADS), (size_t)C::SMEM, stream,
                             PAIR ? 2 : 1, maps.x, maps.w, maps.y, maps.r, a);
}

}  // namespace

static int staging_bytes(int block_n, int pair)
{
    int split = 1, ec = 16;
    tc_epilogue_geometry(block_n, &split, &ec);
    return 4 * tc_epi_warps_per_quarter(block_n, pair != 0) * 2 * 32 * ec * 2;
}

int tc_smem_bytes(int block_n, int block_k, int stages, int pair)
{
    const int a = (kTcBlockM * block_k * 2 + 1023) / 1024 * 1024;
    const int b = ((pair ? block_n / 2 : block_n) * block_k * 2 + 1023) / 1024 * 1024;
    return 1024 + stages * (a + b) + staging_bytes(block_n, pair) + 512;
}

static int stages_for(int block_n, int block_k, int pair = 0)
{
    const int a = (kTcBlockM * block_k * 2 + 1023) / 1024 * 1024;
    const int b = ((pair ? block_n / 2 : block_n) * block_k * 2 + 1023) / 1024 * 1024;
    const int fit = (232448 - 1024 - staging_bytes(block_n, pair) - 512) / (a + b);
    return fit < 8 ? fit : 8;
}

bool tc_supported(const ConvProblem &p)
{
    // TMA needs 16-byte row strides (c % 8, c_out % 8) and the channel chunk of
    // one K step must be one swizzle span of 32/64/128 bytes (c % 16).  The
    // im2col box corners are limited to [-128, 127]; the GEMM row count to int.
    if (p.c % 16 != 0 || p.c_out % 8 != 0) return false;
    if (p.out_fp8 && p.c_out % 16 != 0) return false;  // 16-byte rows of one-byte outputs
    // Square filters with equal stride and padding on both axes only, so the
    // im2col box corners are the same along W and H.
    if (p.r != p.s || p.stride_h != p.stride_w || p.pad_h != p.pad_w) return false;
    if (p.pad_h > 127 || p.pad_w > 127 || p.r - 1 - p.pad_h > 128 || p.s - 1 - p.pad_w > 128) return false;
    if (p.stride_h > 8 || p.stride_w > 8) return false;
    if (p.m > 0x7fffffffLL - kTcBlockM) return false;
    return true;
}

static bool valid_block_n(int bn) { return bn == 16 || bn == 32 || bn == 64 || bn == 128 || bn == 256; }

// Channel-major schedules: the most 128-pixel im2col boxes (per K step) that any
// CTA loads.  Whole tiles: two per tile, tiles dealt round-robin.  Balanced: each
// CTA's equal run of 32-pixel chunks, cut per channel tile into 256-pixel units
// and one remainder (as the kernel's WorkIter cuts them).
static long long swap_boxes_whole(long long tiles, int grid)
{
    return (tiles + grid - 1) / grid * 2;
}

static long long swap_boxes_balanced(long long m, int n_tiles, int grid)
{
    const long long cm = (m + 31) / 32, total = cm * n_tiles;
    long long worst = 0;
    for (int b = 0; b < grid; ++b) {
        long long g = total * b / grid;
        const long long g1 = total * (b + 1) / grid;
        long long boxes = 0;
        while (g < g1) {  // one channel tile's piece of the run per pass
            const long long nt = g / cm;
            const long long pe = std::min(g1, (nt + 1) * cm);
            const long long len = pe - g;
            boxes += len / 8 * 2;
            if (len % 8) {
                const long long p0 = (g + len / 8 * 8 - nt * cm) * 32;
                const long long np = std::min(len % 8 * 32, m - p0);
                boxes += np > kTcBlockM ? 2 : 1;
            }
            g = pe;
        }
        worst = std::max(worst, boxes);
    }
    return worst;
}

int tc_make_plan_request(const ConvProblem &p, int sm_count, const PlanRequest *rq, TcPlan *out)
{
    const PlanRequest dflt{-1, -1, -1, 0, -1, -1, -1};
    const PlanRequest &q = rq ? *rq : dflt;
    if (q.block_n != 0 && !valid_block_n(q.block_n)) return -1;
    TcPlan t{};
    t.block_k = p.c % 64 == 0 ? 64 : (p.c % 32 == 0 ? 32 : 16);
    t.c_chunks = (p.c + t.block_k - 1) / t.block_k;
    t.k_iters = p.r * p.s * t.c_chunks;
    const int m_tiles = (int)((p.m + kTcBlockM - 1) / kTcBlockM);
    const long long tiles256 = (long long)m_tiles * ((p.c_out + 255) / 256);
    if (p.c_out <= 128) {
        t.block_n = p.c_out <= 16 ? 16 : (p.c_out <= 32 ? 32 : (p.c_out <= 64 ? 64 : 128));
    } else if (t.k_iters >= 16 && tiles256 >= sm_count) {
        // Long K loops are tensor-bound: the widest tile (N = 256) moves the fewest
        // shared-memory bytes per MMA, and stream-K (below) evens out the waves.
        t.block_n = 256;
    } else {
        // Choose 128 or 256 output channels per tile by the estimated number of
        // waves times the per-tile work (which scales with the tile width).
        long long best = -1;
        for (int bn : {256, 128}) {
            const long long tiles = (long long)m_tiles * ((p.c_out + bn - 1) / bn);
            const long long waves = (tiles + sm_count - 1) / sm_count;
            const long long cost = waves * bn;
            if (best < 0 || cost < best) {
                best = cost;
                t.block_n = bn;
            }
        }
    }
    // Swap AB for 32..256 output channels: the tile becomes 128 channels x 256
    // pixels so that every MMA runs at N = 256.  Thresholds from a measured sweep
    // of YOLO-shaped layers (the package's tune module): swapped tiles win on
    // 3x3 layers from 32 output channels up and on 1x1 layers from 128, as long
    // as there are tiles for at least half the SMs; they lose where the long-K
    // path above runs 256-wide pair tiles with stream-K, and on 1x1 layers with
    // at most 64 output channels (one or two K steps: the transposing epilogue
    // costs more than the wider MMA saves).
    const long long ptiles256 = (p.m + 255) / 256;
    const long long swap_tiles = ptiles256 * ((p.c_out + kTcBlockM - 1) / kTcBlockM);
    const bool pair_path = p.c_out > 128 && t.k_iters >= 16 && tiles256 >= sm_count;
    const bool short_narrow = p.c_out <= 64 && t.k_iters <= 2;
    // Fewer swap tiles than half the SMs: balanced runs still spread the pixels over
    // every SM, and with K loops of eight steps or more their N = 256-wide MMAs beat
    // the pixel-major tiles (the sweep's 40x40 and 20x20 layers, up to 512 channels;
    // bneck20's 26 swap tiles by 5-11 %, where 128-wide pixel-major tiles keep a third
    // of the SMs busy).  Below an eighth of the SMs (the 1x32x32 layer's 4) the two tie.
    const bool swap_small = p.c_out >= 32 && p.c_out <= 512 && !pair_path && !short_narrow && t.k_iters >= 8 &&
                            swap_tiles >= sm_count / 8 && swap_tiles < sm_count / 2;
    t.swap_ab = ((p.c_out >= 32 && p.c_out <= 256 && !pair_path && !short_narrow && swap_tiles >= sm_count / 2) ||
                 swap_small)
                    ? 1
                    : 0;
    if (q.swap_ab >= 0) t.swap_ab = q.swap_ab ? 1 : 0;
    // Channel-major tiles on the kernel of tc_cmajor.cu: x in tiled boxes of whole output
    // rows (or of the [M][C] matrix of a 1x1 layer) or in im2col boxes; the weights streamed
    // with every K step or resident in tensor memory.
    const bool overrides = q.block_n != 0 || q.stream_k == 1 || q.pair == 1 || q.balanced >= 0 || q.swap_ab == 0;
    if (q.wres == 1 || q.row_boxes == 1) {
        // Requested explicitly.
        TcPlan w{};
        if (overrides) return -1;
        const int wres = q.wres == 1 ? 1 : 0;
        if (q.row_boxes != 0 && cmajor_fill_plan(p, sm_count, wres, 1, &w)) {
            *out = w;
            return 0;
        }
        if (q.row_boxes != 1 && cmajor_fill_plan(p, sm_count, wres, 0, &w)) {
            *out = w;
            return 0;
        }
        return -1;
    }
    if (q.wres < 0 && q.row_boxes < 0 && !overrides) {
        // The planner's own choice, from the measured sweep of YOLO-shaped layers (the package's
        // tune module).  Tiled boxes move at about 1.5x the rate of im2col boxes but only pay
        // with 64-channel K steps (128-byte box rows):
        //  - 1x1 layers read x as a matrix: matrix-row units won or tied on every such layer;
        //  - stride-2 layers of one 64-channel chunk: whole-row units won where they spread as
        //    evenly over the SMs as the im2col runs (the busiest CTA's pixels no more than its
        //    im2col box pixels), and lost by about 10% where they did not (row units come in
        //    whole rows only).  With two or more chunks the im2col runs won (down80: 17.2-17.4
        //    against 18.2-18.4 us), their taps-fastest K order reading one chunk of the input
        //    rows over the first nine steps;
        //  - 3x3 stride-1 layers: im2col runs won on every such layer.
        // With 32-channel K steps on a 3x3 filter and a large layer, im2col units with the
        // weights resident in tensor memory won by 6-28%: the weight tile is a third of each
        // K step's bytes there, and the MMA (A from tensor memory) still has time to spare.
        const bool matrix =
            p.r == 1 && p.s == 1 && p.stride_h == 1 && p.stride_w == 1 && p.pad_h == 0 && p.pad_w == 0;
        TcPlan w{};
        if (t.block_k == 64 && matrix && cmajor_fill_plan(p, sm_count, 0, 1, &w)) {
            *out = w;
            return 0;
        }
        if (t.swap_ab && p.c <= 32 && p.r * p.s >= 9 && p.m >= 256LL * sm_count &&
            cmajor_fill_plan(p, sm_count, 1, 0, &w)) {
            *out = w;
            return 0;
        }
        if (t.swap_ab && t.block_k == 64 && p.c <= 64 && (p.stride_h > 1 || p.stride_w > 1) &&
            cmajor_fill_plan(p, sm_count, 0, 1, &w)) {
            const long long rows_px =
                (long long)(w.m_tiles + w.cm_ctas_per_tile - 1) / w.cm_ctas_per_tile * w.cm_unit_px;
            const int n_ct = (p.c_out + kTcBlockM - 1) / kTcBlockM;
            const long long chunks = (p.m + 31) / 32 * n_ct;
            const long long swap_tiles_all = (p.m + 255) / 256 * n_ct;
            const long long boxes =
                std::min(swap_boxes_balanced(p.m, n_ct, (int)std::min<long long>(chunks, sm_count)),
                         swap_boxes_whole(swap_tiles_all, (int)std::min<long long>(swap_tiles_all, sm_count)));
            if (rows_px <= boxes * kTcBlockM) {
                *out = w;
                return 0;
            }
        }
    }
    if (t.swap_ab) {
        // The channel-major tile is 128 channels x up to 256 pixels.  Whole 256-pixel
        // tiles leave a partly idle last wave (the pointwise layer: 200 tiles on 152
        // SMs); balanced, each CTA instead takes an equal run of the (channel tile,
        // 32-pixel chunk) sequence, cut into units of at most 256 pixels.
        if ((q.block_n != 0 && q.block_n != 256) || q.stream_k == 1 || q.pair == 1) return -1;
        t.block_n = 256;
        t.stages = stages_for(256, t.block_k);
        t.m_tiles = (int)ptiles256;
        t.n_tiles = (p.c_out + kTcBlockM - 1) / kTcBlockM;
        t.tiles = t.m_tiles * t.n_tiles;
        // Balanced runs when they cut the busiest CTA's im2col boxes by a quarter or more
        // (the pointwise layer's 200 tiles put four boxes per K step on 48 CTAs, equal runs
        // at most three on any), or when whole tiles leave SMs idle: equal runs then spread
        // the pixels over every SM (down80's 100 tiles: 17.2-17.4 us balanced against
        // 18.1-18.5 whole, c2f40's 11.9 against 12.5).  Smaller box gains were within the
        // noise of the measured sweep (tune module), and the shorter remainder units cost
        // some of it back.
        const long long chunks = (p.m + 31) / 32 * t.n_tiles;
        const int grid_bal = (int)std::min<long long>(chunks, sm_count);
        const int grid_whole = std::min(t.tiles, sm_count);
        // The kernel splits the chunk sequence with 32-bit arithmetic.
        const bool bal_fits = chunks * grid_bal < (1LL << 32);
        if (q.balanced == 1 && !bal_fits) return -1;
        t.balanced = q.balanced >= 0 ? q.balanced
                                     : (bal_fits && (swap_small || t.tiles < sm_count ||
                                                     4 * swap_boxes_balanced(p.m, t.n_tiles, grid_bal) <=
                                                         3 * swap_boxes_whole(t.tiles, grid_whole))
                                            ? 1
                                            : 0);
        t.grid = t.balanced ? grid_bal : grid_whole;
        t.smem_bytes = tc_smem_bytes(256, t.block_k, t.stages, 0);
        t.stream_k = 0;
        t.pair = 0;
        t.workspace_bytes = 0;
        t.flag_bytes = 0;
        *out = t;
        return 0;
    }
    if (q.balanced == 1) return -1;  // balanced runs are a channel-major schedule
    t.balanced = 0;
    if (q.block_n != 0) t.block_n = q.block_n;
    t.stages = stages_for(t.block_n, t.block_k);
    t.m_tiles = m_tiles;
    t.n_tiles = (p.c_out + t.block_n - 1) / t.block_n;
    t.tiles = t.m_tiles * t.n_tiles;
    t.grid = std::min(t.tiles, sm_count);
    t.smem_bytes = tc_smem_bytes(t.block_n, t.block_k, t.stages, 0);
    // Stream-K when whole tiles would leave a partly idle last wave: every CTA
    // takes total/grid consecutive K steps.  Each share must cover at least one
    // tile so that a tile is split between two CTAs at most.
    const long long total = (long long)t.tiles * t.k_iters;
    // Each share covers at least one tile; the kernel splits the K-step sequence with
    // 32-bit arithmetic.
    const bool sk_possible = total / sm_count >= t.k_iters && total * sm_count < (1LL << 32);
    t.stream_k = (t.tiles > sm_count && t.tiles % sm_count != 0 && t.tiles < 4LL * sm_count &&
                  t.k_iters >= 16 && sk_possible)
                     ? 1
                     : 0;
    if (q.stream_k >= 0) {
        if (q.stream_k == 1 && !sk_possible) return -1;
        t.stream_k = q.stream_k ? 1 : 0;
    }
    if (q.pair == 1 && !t.stream_k) return -1;  // pairs are stream-K workers
    t.workspace_bytes = 0;
    t.flag_bytes = 0;
    t.pair = 0;
    if (t.stream_k) {
        t.grid = sm_count;
        // Pairs of CTAs (clusters of two) run the 2-CTA MMA on pair tiles of
        // 256 x 256, each CTA holding half of the weight tile: the stream-K worker
        // is then the pair.  Each pair's share must cover at least one pair tile.
        const int pair_tiles = (t.m_tiles + 1) / 2 * t.n_tiles;
        const bool pair_possible = t.block_n == 256 && sm_count % 2 == 0 && pair_tiles >= sm_count / 2;
        t.pair = pair_possible ? 1 : 0;
        if (q.pair >= 0) {
            if (q.pair == 1 && !pair_possible) return -1;
            t.pair = q.pair ? 1 : 0;
        }
        if (t.pair) {
            t.tiles = pair_tiles;  // the kernel's work units
            t.stages = stages_for(t.block_n, t.block_k, 1);
            t.smem_bytes = tc_smem_bytes(t.block_n, t.block_k, t.stages, 1);
        }
        const long long slots = t.pair ? (long long)(sm_count / 2 - 1) * 2 : (long long)(t.grid - 1);
        t.flag_bytes = (slots * kTcFlagsPerSlot * (long long)sizeof(int) + 255) / 256 * 256;
        t.workspace_bytes = t.flag_bytes + slots * kTcBlockM * t.block_n * 4;
    }
    *out = t;
    return 0;
}

bool tc_workspace_reserve(cudaStream_t stream)
{
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    for (int i = 0; i < g_ws_count; ++i)
        if (g_ws[i].device == device && g_ws[i].stream == stream) return true;
    if (g_ws_count == kWorkspaceStreams) return false;
    g_ws[g_ws_count++] = Workspace{device, stream, nullptr, 0, 0};
    return true;
}

TcPlan tc_make_plan(const ConvProblem &p, int sm_count)
{
    TcPlan t{};
    tc_make_plan_request(p, sm_count, nullptr, &t);  // the planner's own choices always succeed
    return t;
}

cudaError_t tc_launch(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream)
{
    return tc_launch_with_workspace(p, plan, stream, nullptr);
}

namespace {

template <int EPI>
cudaError_t dispatch(const ConvProblem &p, const TcPlan &plan, const TcMaps &maps, cudaStream_t stream,
                     void *workspace)
{
    if (plan.swap_ab) {
        if (plan.block_n != 256) return cudaErrorInvalidConfiguration;
        if (plan.block_k == 64) return launch_cfg<256, 64, true, false, EPI>(p, plan, maps, stream, workspace);
        if (plan.block_k == 32) return launch_cfg<256, 32, true, false, EPI>(p, plan, maps, stream, workspace);
        if (plan.block_k == 16) return launch_cfg<256, 16, true, false, EPI>(p, plan, maps, stream, workspace);
        return cudaErrorInvalidConfiguration;
    }
    if (plan.pair) {
        if (plan.block_n != 256) return cudaErrorInvalidConfiguration;
        if (plan.block_k == 64) return launch_cfg<256, 64, false, true, EPI>(p, plan, maps, stream, workspace);
        if (plan.block_k == 32) return launch_cfg<256, 32, false, true, EPI>(p, plan, maps, stream, workspace);
        if (plan.block_k == 16) return launch_cfg<256, 16, false, true, EPI>(p, plan, maps, stream, workspace);
        return cudaErrorInvalidConfiguration;
    }
#define CBS_TC_CASE(BN_, BK_) \
    if (plan.block_n == BN_ && plan.block_k == BK_)       \
        return launch_cfg<BN_, BK_, false, false, EPI>(p, plan, maps, stream, workspace);
    CBS_TC_CASE(16, 16) CBS_TC_CASE(16, 32) CBS_TC_CASE(16, 64)
    CBS_TC_CASE(32, 16) CBS_TC_CASE(32, 32) CBS_TC_CASE(32, 64)
    CBS_TC_CASE(64, 16) CBS_TC_CASE(64, 32) CBS_TC_CASE(64, 64)
    CBS_TC_CASE(128, 16) CBS_TC_CASE(128, 32) CBS_TC_CASE(128, 64)
    CBS_TC_CASE(256, 16) CBS_TC_CASE(256, 32) CBS_TC_CASE(256, 64)
#undef CBS_TC_CASE
    return cudaErrorInvalidConfiguration;
}

}  // namespace

cudaError_t tc_launch_with_workspace(const ConvProblem &p, const TcPlan &plan, cudaStream_t stream,
                                     void *workspace)
{
    if (plan.cmajor) return cmajor_launch(p, plan, stream);
    TcMaps maps;
    cudaError_t st = cached_maps(p, plan.block_n, plan.block_k, plan.swap_ab != 0, plan.pair != 0, &maps);
    if (st != cudaSuccess) return st;
    if (p.out_fp8) {
        if (p.residual != nullptr) return cudaErrorInvalidConfiguration;
        return dispatch<kEpiKindFp8>(p, plan, maps, stream, workspace);
    }
    if (p.residual != nullptr) {
        // The residual's map changes with its pointer: encoded per call (a host call
        // of a few microseconds, next to the cached maps).
        st = encode_bf16_like_y(p, plan.block_n, plan.swap_ab != 0, p.residual, &maps.r);
        if (st != cudaSuccess) return st;
        return dispatch<kEpiKindResidual>(p, plan, maps, stream, workspace);
    }
    if (p.epi_mode != kEpiSilu) return dispatch<kEpiKindMode>(p, plan, maps, stream, workspace);
    return dispatch<kEpiKindSilu>(p, plan, maps, stream, workspace);
}

cudaError_t tc_reset_workspaces()
{
    std::lock_guard<std::mutex> lock(g_ws_mu);
    int prev = 0;
    cudaError_t st = cudaGetDevice(&prev);
    if (st != cudaSuccess) return st;
    for (int i = 0; i < g_ws_count && st == cudaSuccess; ++i) {
        if (!g_ws[i].ptr) continue;
        st = cudaSetDevice(g_ws[i].device);
        if (st == cudaSuccess) st = cudaStreamSynchronize(g_ws[i].stream);
        if (st == cudaSuccess) st = cudaMemset(g_ws[i].ptr, 0, g_ws[i].flag_bytes);
    }
    cudaSetDevice(prev);
    return st;
}

cudaError_t tc_read_and_clear_error(cudaStream_t stream, unsigned int *out)
{
    unsigned int host = 0;
    cudaError_t st = cudaMemcpyFromSymbolAsync(&host, g_tc_error, sizeof host, 0,
                                               cudaMemcpyDeviceToHost, stream);
    if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    if (st != cudaSuccess) return st;
    if (host != 0) {
        const unsigned int zero = 0;
        st = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
        if (st == cudaSuccess) st = cudaStreamSynchronize(stream);
    }
    *out = host;
    return st;
}

}  // namespace cbs
