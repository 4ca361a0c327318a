// hc_pre_wide.cu -- the pre-chain for 5 <= s <= 8 streams, on every SM of the GPU.
//
// What it computes (memra-engine hyper.rs page, module header "ARITHMETIC
// CONTRACT"): per token, mixes = fn_w . x[t] over the whole s*d slab, rescaled by
// rsqrt(mean(x[t]^2) + eps); the pre/post gates and the Sinkhorn comb from the
// logits mixes*scale[group] + base; the collapse y[t] = sum_c pre_c x[t,c].
//
// Why a separate kernel: at s = 8, d = 7168 (rows R = 80, K = s*d = 57344) the
// contraction is ~36 FLOP per byte of x, so float32 FMA throughput decides the
// time, and fn_w (17.5 MiB) is far too large for one SM.  So every CTA of one
// persistent grid (one CTA per SM) keeps a fixed K slice of fn_w resident:
//
//  * CTA b owns hidden columns [h0_b, h0_b + hw_b) of every stream (hw_b a multiple
//    of 8 with s*hw_b % 64 == 0; widths differ by at most one unit), i.e. an LK =
//    s*hw_b column slice of each token's slab and the matching LK columns of all R
//    rows of fn_w, which sit in tensor memory (TMEM, used as per-thread storage)
//    for the whole launch.  Every CTA sees every token.
//  * Token tiles of kWM tokens arrive by one 3-D TMA load (box hw_b x s x kWM) into a
//    deep ring of shared-memory stages (a tile's slice is only a few KiB), so x is
//    read from HBM once.
//  * Eight compute warps: warp w owns rows [B*w, B*w+B) (B = ceil(R/8)); its 32
//    lanes are K-groups, lane l owning columns 2l, 2l+1 of every 64-column group
//    of the slice; every warp does all kWM tokens of a tile.  Packed float32 FMAs
//    (x from shared memory, fn_w from TMEM), a 32-lane xor reduce-scatter, and the
//    tile's partial dots and sums of squares go to a slot of the workspace.
//  * A publisher warp raises the tile's counter once the CTA's eight compute warps
//    have written their partials of the tile.
//  * Tiles are finished by fixed, rotating CTAs (no CTA's share of the work depends
//    on its timing), in two steps: each of the 4*RV/4 float4 columns of a tile's
//    partial rows has a reducer CTA, which sums that column over every CTA's row
//    (lanes over rows, then a fixed xor tree: one round trip to L2); the tile's
//    finisher gathers the reduced columns, forms the gates (pre and post written
//    out), sets the tile's flag and then runs the tile's Sinkhorn.  Each CTA has one
//    warp for each step; each takes its duties in tile order and waits (bounded) for
//    the counters they need.
//  * A collapse warp in every CTA waits (bounded) for each tile's flag, writes y
//    for the CTA's hidden columns from the stage, and refills the stage.  The compute
//    warps wait only for stages, so the ring is the only way later tiles wait for
//    earlier ones; no wait depends on a later tile, so the grid cannot deadlock.
//  * Every wait is bounded (2 s); on timeout the kernel records the site in the
//    workspace status word and winds down.  The host zeroes the tiles' counters and
//    flags (a memset on the stream) before each launch, so what other paths or
//    earlier calls left in the workspace does not matter.
//
// Determinism: every partial has a fixed summation order (per lane, then the xor
// tree), the partials of a token are summed over CTAs in a fixed order (within each
// group, then over groups), and no float atomics are used: repeated calls give the
// same bits, and a token's results do not depend on the other tokens of the batch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "hc_internal.cuh"
#include "hc_ptx.cuh"

namespace hc {
namespace {

constexpr int kWThreads = 384;            // 12 warps
constexpr int kWNCW = 8;                  // compute warps 0-7, one row group each
constexpr int kWPublishWarp = 8;          // counts this CTA's partials into its group's counter
constexpr int kWReduceWarp = 9;           // column sums of the (tile, column) pairs this CTA reduces
constexpr int kWTileWarp = 10;            // tile finishes (gates, flag, Sinkhorn) of this CTA's tiles
constexpr int kWCollapseWarp0 = 11;       // warp 11: collapse and stage refills
constexpr int kWM = 4;                    // tokens per tile
constexpr int kWNst = 24;                 // stages of the ring = partial slots
constexpr int kWMaxCtas = 160;            // workspace sizing bound on the grid
constexpr uint32_t kWTmemCols = 256;
constexpr int kWMaxTmemCols = 256;
constexpr unsigned long long kWWaitNs = 2000000000ull;
constexpr uint32_t kNbWCompute = 1;       // named barrier of the compute warps
constexpr unsigned kFullMask = 0xffffffffu;

enum WSite : unsigned { kWSiteW = 32, kWSiteFull, kWSiteShipped, kWSiteFlag, kWSiteReduce, kWSiteTile, kWSiteDrain };

template <int S>
struct WG {
    static constexpr int R = (2 + S) * S;
    static constexpr int B = (R + kWNCW - 1) / kWNCW;      // rows per compute warp
    static constexpr int WB = (2 * B + 3) / 4 * 4;          // TMEM columns per 64-column group
    static constexpr int RV = R + 1;                         // partial values per token: R dots + sum of squares
    static constexpr int NV = kWM * B + 1;                   // per-lane values before the reduce-scatter
    static constexpr int NVP = (NV + 31) / 32 * 32;
    static constexpr int VPL = NVP / 32;                     // per-lane values after it
};

struct WParams {
    CUtensorMap tmap_x[2];   // x as (d, s, T), box (hw[i], s, kWM)
    CUtensorMap tmap_w[2];   // fn_w as (d, s, R), box (hw[i], s, R)
    const float *scale, *base;
    float *pre, *post, *comb, *y;
    StatusBlock *status;
    unsigned *pcount;   // [ntiles]: CTAs whose partials of the tile are out (zero at launch)
    unsigned *tcount;   // [ntiles]: reduced columns of the tile written (zero at launch)
    unsigned *flags;    // [ntiles]: the tile's gates are out (zero at launch)
    float *part;        // [kWNst][ncta][kWM][RV]: each CTA's partials of a tile
    float *red;         // [kWNst][kWM][RV]: the tile's sums over every CTA
    int T, d, ntiles, ncta, iters;
    int nwide, hw0, hw1;   // CTAs [0, nwide) own hw0 columns, the rest hw1
    float eps, invK;       // invK = 1 / (s*d)
    unsigned long long *stamps;   // phase stamps (HC_STAMPS builds), else null
};

// Phase stamps (HC_STAMPS builds only).  Slot 0: CTA 0's compute warp 0
// (kEvStageReady, kEvDotsDone, kEvShipped), publisher (kEvPartials) and collapse warp
// (kEvPreArrived, kEvCollapsed, kEvRefilled).  Slot 1, whichever CTA does it: the
// reduction of column 0 of each tile (kEvXfStart: every CTA's partials out, kEvXfDone:
// column sum written) and each tile's finish (kEvXfLanded: every column in,
// kEvGatesSent: flag set, kEvSinkDone).
#ifdef HC_STAMPS
__device__ __forceinline__ void w_stamp_at(const WParams &p, int slot, int it, int ev)
{
    if (p.stamps && (slot == 1 || blockIdx.x == 0) && it >= 0 && it < kStampTiles)
        p.stamps[((size_t)slot * kStampTiles + it) * kStampEvents + ev] = ptx::globaltimer();
}
#define W_STAMP(it, ev) w_stamp_at(p, 0, (it), (ev))
#define W_STAMP_ANY(it, ev) w_stamp_at(p, 1, (it), (ev))
#else
#define W_STAMP(it, ev) \
    do {                \
    } while (0)
#define W_STAMP_ANY(it, ev) \
    do {                    \
    } while (0)
#endif

struct WLay {
    int stage_bytes, off_red, off_ex, off_bar, off_misc, total;
};

template <int S>
__host__ __device__ inline WLay make_wlay(int lk_max)
{
    WLay L;
    L.stage_bytes = kWM * lk_max * 4;
    int o = kWNst * L.stage_bytes;
    L.off_red = o;                   // [kWM][RV]: the finished tile's summed partials
    o += kWM * WG<S>::RV * 4;
    o = (o + 15) / 16 * 16;
    L.off_ex = o;                    // [kWM][S*S]: the finished tile's exp(comb logits),
    o += kWM * S * S * 4;            // then [kWM][S]: the collapse warp's copy of a tile's pre gates
    o += kWM * S * 4;
    L.off_bar = o;                   // full[kWNst], shipped[kWNst], wfull
    o += (2 * kWNst + 1) * 8;
    L.off_misc = o;                  // TMEM address, abort flag, TMA loads issued per stage
    o += 16 + kWNst * 4;
    L.total = (o + 127) / 128 * 128;
    return L;
}

__device__ __forceinline__ void w_report(StatusBlock *sb, unsigned site)
{
    if (atomicCAS(&sb->code, 0u, (unsigned)kDevWaitTimeout) == 0u) {
        sb->where = site;
        sb->block = blockIdx.x;
    }
}

// Bounded wait on an mbarrier phase of this CTA (see the cluster kernel's wait_bar).
__device__ __forceinline__ bool w_wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           StatusBlock *sb, unsigned site, bool honor_abort = true)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((n & 63u) == 0u) {
            if (honor_abort) {
                if (*abort_flag)
                    return false;
                if (*reinterpret_cast<volatile unsigned *>(&sb->code) != 0u) {
                    *abort_flag = 1;
                    return false;
                }
            }
            if (ptx::globaltimer() - t0 > kWWaitNs) {
                w_report(sb, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool w_warp_wait(int lane, uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            StatusBlock *sb, unsigned site)
{
    bool ok = true;
    if (lane == 0)
        ok = w_wait_bar(bar, parity, abort_flag, sb, site);
    ok = __shfl_sync(kFullMask, ok, 0);
    __syncwarp();
    return ok;
}

// Bounded poll of a counter that other CTAs raise, until it reaches `target` (acquire).
__device__ __forceinline__ bool w_wait_count(const unsigned *ctr, unsigned target, volatile int *abort_flag,
                                             StatusBlock *sb, unsigned site)
{
    if (ptx::ld_acquire_gpu(ctr) >= target)
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        ptx::nanosleep(64);
        if (ptx::ld_acquire_gpu(ctr) >= target)
            return true;
        if ((n & 15u) == 0u) {
            if (*abort_flag)
                return false;
            if (*reinterpret_cast<volatile unsigned *>(&sb->code) != 0u) {
                *abort_flag = 1;
                return false;
            }
            if (ptx::globaltimer() - t0 > kWWaitNs) {
                w_report(sb, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Bounded wait by lane 0 of a warp for a counter; every lane gets the answer and can
// read what the counter's raisers wrote before it.
__device__ __forceinline__ bool w_warp_wait_count(int lane, const unsigned *ctr, unsigned target,
                                                  volatile int *abort_flag, StatusBlock *sb, unsigned site)
{
    bool ok = true;
    if (lane == 0)
        ok = w_wait_count(ctr, target, abort_flag, sb, site);
    ok = __shfl_sync(kFullMask, ok, 0);
    __threadfence();
    return ok;
}

// One level of the xor reduce-scatter over the 32 lanes of a warp (lanes whose M bit
// is clear keep the lower half of the list and add their partner's copy of it).
template <int N, int M>
__device__ __forceinline__ void w_rs_level(float *v, int lane)
{
    constexpr int H = N / 2;
    const bool hi = (lane & M) != 0;
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const float a = v[k], b = v[k + H];
        const float send = hi ? a : b;
        const float keep = hi ? b : a;
        v[k] = keep + __shfl_xor_sync(kFullMask, send, M);
    }
}
// After it, lane l holds the warp sums of values [VPL*l, VPL*l + VPL) (N = 32 * VPL).
template <int N>
__device__ __forceinline__ void w_reduce_scatter32(float *v, int lane)
{
    w_rs_level<N, 16>(v, lane);
    w_rs_level<N / 2, 8>(v, lane);
    w_rs_level<N / 4, 4>(v, lane);
    w_rs_level<N / 8, 2>(v, lane);
    w_rs_level<N / 16, 1>(v, lane);
}

template <int N>
__device__ __forceinline__ float w_tree_sum(const float *v)
{
    if constexpr (N == 1) {
        return v[0];
    } else {
        return w_tree_sum<N / 2>(v) + w_tree_sum<N - N / 2>(v + N / 2);
    }
}

// Sinkhorn on an S x S matrix in registers: `iters` rounds of dividing each row by
// (row sum + eps), then each column by (column sum + eps), with correctly rounded
// reciprocals.
template <int S>
__device__ __forceinline__ void w_sinkhorn(float *c, int iters, float eps)
{
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const float inv = 1.0f / (w_tree_sum<S>(c + j * S) + eps);
#pragma unroll
            for (int k = 0; k < S; ++k)
                c[j * S + k] *= inv;
        }
#pragma unroll
        for (int k = 0; k < S; ++k) {
            float col[S];
#pragma unroll
            for (int j = 0; j < S; ++j)
                col[j] = c[j * S + k];
            const float inv = 1.0f / (w_tree_sum<S>(col) + eps);
#pragma unroll
            for (int j = 0; j < S; ++j)
                c[j * S + k] *= inv;
        }
    }
}

template <int S>
__global__ void __launch_bounds__(kWThreads, 1) hc_pre_wide_kernel(const __grid_constant__ WParams p)
{
    using G = WG<S>;
    constexpr int R = G::R, B = G::B, WB = G::WB, RV = G::RV;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int hw = cta < p.nwide ? p.hw0 : p.hw1;
    const int h0 = cta < p.nwide ? cta * p.hw0 : p.nwide * p.hw0 + (cta - p.nwide) * p.hw1;
    const int LK = S * hw, NJ = LK / 64;
    const WLay L = make_wlay<S>(S * p.hw0);
    const CUtensorMap *tmx = &p.tmap_x[cta < p.nwide ? 0 : 1];
    const CUtensorMap *tmw = &p.tmap_w[cta < p.nwide ? 0 : 1];
    float *stages = reinterpret_cast<float *>(smem);
    float *red = reinterpret_cast<float *>(smem + L.off_red);
    float *ex = reinterpret_cast<float *>(smem + L.off_ex);
    const uint32_t bar0 = ptx::smem_u32(smem + L.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L.off_misc + 16);   // per stage
    StatusBlock *sb = p.status;
    const int stage_floats = L.stage_bytes / 4;
    auto FULL = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto SHIPPED = [&](int s) { return bar0 + 8u * (uint32_t)(kWNst + s); };
    const uint32_t WFULL = bar0 + 8u * (uint32_t)(2 * kWNst);
    const uint32_t tile_bytes = (uint32_t)(kWM * LK * 4);
    auto load_tile = [&](int it) {   // one thread; the stage must be free
        const int s = it % kWNst;
        ptx::mbar_arrive_expect_tx(FULL(s), tile_bytes);
        ptx::tma_load_3d(ptx::smem_u32(stages + s * stage_floats), tmx, h0, 0, it * kWM, FULL(s));
        issued[s] = issued[s] + 1;
    };

    // ------------------------------------------------------------------ set-up
    if (threadIdx.x == 0)
        W_STAMP(0, kEvKernelStart);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kWNst; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(SHIPPED(s), kWNCW);   // every compute warp arrives once per tile
            issued[s] = 0;
        }
        ptx::mbar_init(WFULL, 1);
        // A non-zero status word (an earlier launch timed out) makes this launch skip its
        // work; the word can only change 2 s into a launch, so every CTA reads the same.
        *abort_flag = *reinterpret_cast<volatile unsigned *>(&sb->code) != 0u ? 1 : 0;
        ptx::fence_mbar_init_cluster();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kWTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tmem_fence_before_sync();
    __syncthreads();
    ptx::tmem_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const bool skip = *abort_flag != 0;

    if (!skip && warp < kWNCW) {
        // -------------------------------------------------------------- compute warps
        const int sp = warp & 3;
        const uint32_t trow = tmem_base + ((uint32_t)(32 * sp) << 16) + (uint32_t)((warp >> 2) * WB * NJ);
        if (threadIdx.x == 0) {   // this CTA's fn_w slice, staged through the stage ring
            ptx::prefetch_tmap(tmx);
            ptx::prefetch_tmap(tmw);
            ptx::mbar_arrive_expect_tx(WFULL, (uint32_t)(R * LK * 4));
            ptx::tma_load_3d(ptx::smem_u32(stages), tmw, h0, 0, 0, WFULL);
        }
        bool ok = w_warp_wait(lane, WFULL, 0, abort_flag, sb, kWSiteW);
        if (ok) {
            // This lane's fn_w values -> its TMEM lane: column group jj at columns
            // jj*WB .., row r's column pair (2l, 2l+1 of the group) at 2r, 2r+1.
            const float *wst = stages;
            for (int jj = 0; jj < NJ; ++jj) {
                float a[WB];
#pragma unroll
                for (int r = 0; r < B; ++r) {
                    const int row = warp * B + r;
                    float2 v = make_float2(0.f, 0.f);
                    if (row < R)
                        v = *reinterpret_cast<const float2 *>(wst + row * LK + 64 * jj + 2 * lane);
                    a[2 * r] = v.x;
                    a[2 * r + 1] = v.y;
                }
#pragma unroll
                for (int q = 2 * B; q < WB; ++q)
                    a[q] = 0.f;
#pragma unroll
                for (int m = 0; m < WB / 4; ++m)
                    ptx::tmem_st4(trow + (uint32_t)(jj * WB + 4 * m), a + 4 * m);
            }
            ptx::tmem_wait_st();
        }
        ptx::tmem_fence_before_sync();
        ok = ptx::named_bar_and(kNbWCompute, kWNCW * 32, ok);   // the staged slice may be overwritten
        ptx::tmem_fence_after_sync();
        if (ok && threadIdx.x == 0)
            for (int it = 0; it < kWNst && it < p.ntiles; ++it)
                load_tile(it);
        for (int it = 0; ok && it < p.ntiles; ++it) {
            const int s = it % kWNst;
            if (!(ok = w_warp_wait(lane, FULL(s), (it / kWNst) & 1, abort_flag, sb, kWSiteFull)))
                break;
            if (threadIdx.x == 0)
                W_STAMP(it, kEvStageReady);
            const uint32_t xs = ptx::smem_u32(stages + s * stage_floats) + 8u * (uint32_t)lane;
            float2 acc[kWM][B];
            float2 ssa = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kWM; ++i)
#pragma unroll
                for (int r = 0; r < B; ++r)
                    acc[i][r] = make_float2(0.f, 0.f);
            for (int jj = 0; jj < NJ; ++jj) {
                float2 xp[kWM];
                float w[WB];
#pragma unroll
                for (int i = 0; i < kWM; ++i)
                    xp[i] = ptx::lds64(xs + (uint32_t)(i * LK * 4 + jj * 256));
                ptx::tmem_ld_issue<WB>(trow + (uint32_t)(jj * WB), w);
                ptx::tmem_ld_wait_regs<WB>(w);
#pragma unroll
                for (int i = 0; i < kWM; ++i)
#pragma unroll
                    for (int r = 0; r < B; ++r)
                        acc[i][r] = ptx::ffma2(xp[i], make_float2(w[2 * r], w[2 * r + 1]), acc[i][r]);
                // Warp w also sums the squares of the tile's token w (w < kWM).
#pragma unroll
                for (int i = 0; i < kWM; ++i)
                    if (i == warp)
                        ssa = ptx::ffma2(xp[i], xp[i], ssa);
            }
            if (threadIdx.x == 0)
                W_STAMP(it, kEvDotsDone);
            float v[G::NVP];
#pragma unroll
            for (int i = 0; i < kWM; ++i)
#pragma unroll
                for (int r = 0; r < B; ++r)
                    v[i * B + r] = acc[i][r].x + acc[i][r].y;
            v[kWM * B] = ssa.x + ssa.y;
#pragma unroll
            for (int q = G::NV; q < G::NVP; ++q)
                v[q] = 0.f;
            w_reduce_scatter32<G::NVP>(v, lane);
            // This CTA's partials of the tile -> slot it % kWNst: [token][R dots, squares].
            float *dst = p.part + ((size_t)s * p.ncta + cta) * kWM * RV;
#pragma unroll
            for (int q = 0; q < G::VPL; ++q) {
                const int o = G::VPL * lane + q;
                if (o < kWM * B) {
                    const int i = o / B, row = warp * B + (o - (o / B) * B);
                    if (row < R)
                        dst[i * RV + row] = v[q];
                } else if (o == kWM * B && warp < kWM) {
                    dst[warp * RV + R] = v[q];
                }
            }
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(SHIPPED(s));   // release: the publisher warp publishes them
            if (threadIdx.x == 0)
                W_STAMP(it, kEvShipped);
        }
    } else if (!skip && warp == kWPublishWarp) {
        // -------------------------------------------------------------- publisher warp
        // Once this CTA's eight compute warps have written a tile's partials, raise the
        // tile's counter (one fence covers every tile found ready).
        int it = 0;
        while (it < p.ntiles) {
            if (!w_warp_wait(lane, SHIPPED(it % kWNst), (it / kWNst) & 1, abort_flag, sb, kWSiteShipped))
                break;
            int last = it;
            while (last + 1 < p.ntiles && last + 1 < it + kWNst &&
                   ptx::mbar_test_wait(SHIPPED((last + 1) % kWNst), ((last + 1) / kWNst) & 1))
                ++last;
            if (lane == 0) {
                __threadfence();
                for (int k = it; k <= last; ++k) {
                    atomicAdd(&p.pcount[k], 1u);
                    W_STAMP(k, kEvPartials);
                }
            }
            __syncwarp();
            it = last + 1;
        }
    } else if (!skip && (warp == kWReduceWarp || warp == kWTileWarp)) {
        // -------------------------------------------------------------- finisher warps
        // Reduce warp: the column sums of the (tile, column) pairs this CTA reduces,
        // column q of tile it going to CTA (it*Q4 + q) % ncta.  Tile warp: the finish of
        // the tiles this CTA owns (tile it to CTA it % ncta).  Each takes its duties in
        // tile order.
        constexpr int Q4 = kWM * RV / 4;
        static_assert((kWM * RV) % 4 == 0, "partial rows are whole float4s");
        const bool reduce_role = warp == kWReduceWarp;
        if (reduce_role) {
            // Pairs (it, q) with (it*Q4 + q) % ncta == cta, in order of it then q.
            for (int it = 0; it < p.ntiles; ++it) {
                const int base = (int)(((long long)it * Q4) % p.ncta);
                int q = cta - base;
                if (q < 0)
                    q += p.ncta;
                if (q >= Q4)
                    continue;
                if (!w_warp_wait_count(lane, &p.pcount[it], (unsigned)p.ncta, abort_flag, sb, kWSiteReduce))
                    break;
                if (lane == 0 && q == 0)
                    W_STAMP_ANY(it, kEvXfStart);
                const int s = it % kWNst;
                const float4 *src = reinterpret_cast<const float4 *>(p.part + (size_t)s * p.ncta * kWM * RV);
                float4 *dst = reinterpret_cast<float4 *>(p.red + (size_t)s * kWM * RV);
                for (; q < Q4; q += p.ncta) {
                    // lane l sums rows l, l+32, ... in row order; then a fixed xor tree
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                    float4 v[(kWMaxCtas + 31) / 32];
#pragma unroll
                    for (int m = 0; m < (kWMaxCtas + 31) / 32; ++m) {
                        const int c = lane + 32 * m;
                        v[m] = c < p.ncta ? __ldcg(src + (size_t)c * Q4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int m = 0; m < (kWMaxCtas + 31) / 32; ++m) {
                        if (lane + 32 * m < p.ncta) {
                            a.x += v[m].x;
                            a.y += v[m].y;
                            a.z += v[m].z;
                            a.w += v[m].w;
                        }
                    }
#pragma unroll
                    for (int mask = 16; mask >= 1; mask >>= 1) {
                        a.x += __shfl_xor_sync(kFullMask, a.x, mask);
                        a.y += __shfl_xor_sync(kFullMask, a.y, mask);
                        a.z += __shfl_xor_sync(kFullMask, a.z, mask);
                        a.w += __shfl_xor_sync(kFullMask, a.w, mask);
                    }
                    if (lane == 0)
                        dst[q] = a;
                }
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    // the number of this CTA's columns of the tile
                    int nq = 0;
                    for (int qq = cta - base < 0 ? cta - base + p.ncta : cta - base; qq < Q4; qq += p.ncta)
                        ++nq;
                    atomicAdd(&p.tcount[it], (unsigned)nq);
                    if (cta == base)
                        W_STAMP_ANY(it, kEvXfDone);
                }
                __syncwarp();
            }
        } else {
        for (int it = cta; it < p.ntiles; it += p.ncta) {
            const int s = it % kWNst;
            // tile finish: gather the column sums, the gates, the flag, the Sinkhorn
            if (!w_warp_wait_count(lane, &p.tcount[it], (unsigned)Q4, abort_flag, sb, kWSiteTile))
                break;
            if (lane == 0)
                W_STAMP_ANY(it, kEvXfLanded);
            const float4 *src = reinterpret_cast<const float4 *>(p.red + (size_t)s * kWM * RV);
            for (int q = lane; q < Q4; q += 32)
                reinterpret_cast<float4 *>(red)[q] = __ldcg(src + q);
            __syncwarp();
            const int t0 = it * kWM, tm = min(kWM, p.T - t0);
            for (int e = lane; e < tm * R; e += 32) {
                const int i = e / R, r = e - (e / R) * R;
                const float rinv = rsqrtf(red[i * RV + R] * p.invK + p.eps);
                const int grp = r < S ? 0 : (r < 2 * S ? 1 : 2);
                const float logit = red[i * RV + r] * rinv * p.scale[grp] + p.base[r];
                if (r < 2 * S) {
                    const float sg = 1.f / (1.f + expf(-logit));
                    if (r < S)
                        p.pre[(size_t)(t0 + i) * S + r] = sg + p.eps;
                    else
                        p.post[(size_t)(t0 + i) * S + (r - S)] = 2.f * sg;
                } else {
                    ex[i * S * S + (r - 2 * S)] = expf(logit);
                }
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence();                      // pre is visible before the flag
                ptx::st_release_gpu(&p.flags[it], 1u);
                W_STAMP_ANY(it, kEvGatesSent);
            }
            // The tile's Sinkhorn, one token per lane (this warp's next tile is ncta tiles on).
            if (lane < tm) {
                float cm[S * S];
#pragma unroll
                for (int q = 0; q < S * S; ++q)
                    cm[q] = ex[lane * S * S + q];
                w_sinkhorn<S>(cm, p.iters, p.eps);
                float *dst = p.comb + (size_t)(t0 + lane) * S * S;
#pragma unroll
                for (int q = 0; q < S * S; ++q)
                    dst[q] = cm[q];
            }
            __syncwarp();
            if (lane == 0)
                W_STAMP_ANY(it, kEvSinkDone);
        }
        }
    } else if (!skip && warp >= kWCollapseWarp0) {
        // -------------------------------------------------------------- collapse warp
        // Tile by tile: wait for the tile's flag, load its pre gates once (one lane per
        // token and stream), write y for this CTA's hidden columns from the stage, then
        // refill the stage with tile it + kWNst.
        const int h4n = hw / 4;
        float *pre_s = ex + kWM * S * S;   // [kWM][S]: the collapse warp's own copy of the tile's gates
        static_assert(kWM * S <= 32, "one lane per gate of the tile");
        for (int it = 0; it < p.ntiles; ++it) {
            if (!w_warp_wait_count(lane, &p.flags[it], 1u, abort_flag, sb, kWSiteFlag))
                break;
            if (lane == 0)
                W_STAMP(it, kEvPreArrived);
            const int s = it % kWNst;
            const int t0 = it * kWM, tm = min(kWM, p.T - t0);
            if (lane < tm * S)
                pre_s[lane] = __ldcg(p.pre + (size_t)t0 * S + lane);
            __syncwarp();
            const float *xs = stages + s * stage_floats;
            for (int e = lane; e < tm * h4n; e += 32) {
                const int i = e / h4n, c4 = e - (e / h4n) * h4n;
                const float *pr = pre_s + i * S;
                const float *xr = xs + i * LK + 4 * c4;
                float4 xv = *reinterpret_cast<const float4 *>(xr);
                float4 a = make_float4(pr[0] * xv.x, pr[0] * xv.y, pr[0] * xv.z, pr[0] * xv.w);
#pragma unroll
                for (int k = 1; k < S; ++k) {
                    xv = *reinterpret_cast<const float4 *>(xr + k * hw);
                    a.x = fmaf(pr[k], xv.x, a.x);
                    a.y = fmaf(pr[k], xv.y, a.y);
                    a.z = fmaf(pr[k], xv.z, a.z);
                    a.w = fmaf(pr[k], xv.w, a.w);
                }
                *reinterpret_cast<float4 *>(p.y + (size_t)(t0 + i) * p.d + h0 + 4 * c4) = a;
            }
            __syncwarp();
            if (lane == 0) {
                W_STAMP(it, kEvCollapsed);
                if (it + kWNst < p.ntiles) {
                    load_tile(it + kWNst);
                    W_STAMP(it, kEvRefilled);
                }
            }
            __syncwarp();
        }
    }

    // ------------------------------------------------------------------ teardown
    ptx::tmem_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        // Every TMA load this CTA issued lands before it exits.
        if (!skip)
            w_wait_bar(WFULL, 0, abort_flag, sb, kWSiteDrain, false);
        for (int s = 0; s < kWNst; ++s)
            if (issued[s] > 0)
                w_wait_bar(FULL(s), (issued[s] - 1) & 1, abort_flag, sb, kWSiteDrain, false);
    }
    __syncthreads();
    ptx::tmem_fence_after_sync();
    if (warp == 0)
        ptx::tmem_dealloc(tmem_base, kWTmemCols);
}

// ---------------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 w_encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

// Map a row-major [rows][s][d] float tensor as (d, s, rows) with a box (hw, s, box_rows);
// reads past the last row are zero-filled.
bool w_encode(CUtensorMap *m, const float *base, int rows, int s, int d, int hw, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = w_encode_fn();
    if (!enc)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)s * d * 4};   // bytes
    const cuuint32_t box[3] = {(cuuint32_t)hw, (cuuint32_t)s, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The hidden split: widths are multiples of the unit u (the smallest multiple of 8 with
// s*u % 64 == 0), at most one unit apart, over as many CTAs as the device has SMs.
struct WideSplit {
    int ncta = 0, nwide = 0, hw0 = 0, hw1 = 0;
};

int wide_unit(int s)
{
    for (int u = 8;; u += 8)
        if ((s * u) % 64 == 0)
            return u;
}

template <int S>
bool wide_split_for(int d, int nsm, int max_smem, WideSplit &w)
{
    using G = WG<S>;
    const int u = wide_unit(S);
    if (d % u != 0 || nsm < 1)
        return false;
    const int units = d / u;
    const int ncta = units < nsm ? units : nsm;
    const int per = units / ncta, extra = units % ncta;
    w.ncta = ncta;
    w.nwide = extra ? extra : ncta;
    w.hw0 = (per + (extra ? 1 : 0)) * u;
    w.hw1 = per * u;
    const int lk_max = S * w.hw0;
    if (lk_max % 64 != 0 || w.hw0 > 256)
        return false;
    if (2 * G::WB * (lk_max / 64) > kWMaxTmemCols)   // two compute warps share each TMEM lane
        return false;
    if (G::R * lk_max > kWNst * kWM * lk_max)        // the fn_w slice is staged through the ring
        return false;
    if (make_wlay<S>(lk_max).total > max_smem)
        return false;
    // Enough CTAs to be worth a whole-GPU launch, and the widths balanced to 3/4.
    if (ncta < 32 || (double)units / ((double)ncta * (per + (extra ? 1 : 0))) < 0.75)
        return false;
    return true;
}

bool wide_split(int s, int d, const DeviceInfo &di, WideSplit &w)
{
    switch (s) {
    case 5: return wide_split_for<5>(d, di.sm_count, di.max_smem_optin, w);
    case 6: return wide_split_for<6>(d, di.sm_count, di.max_smem_optin, w);
    case 7: return wide_split_for<7>(d, di.sm_count, di.max_smem_optin, w);
    case 8: return wide_split_for<8>(d, di.sm_count, di.max_smem_optin, w);
    default: return false;
    }
}

struct WideInfo {
    unsigned long long ctx = 0;
    bool ok = false;
};

template <int S>
bool wide_ready(const DeviceInfo &di)
{
    static std::mutex mu;
    static WideInfo info[64];
    if (di.device < 0 || di.device >= 64)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    WideInfo &wi = info[di.device];
    const unsigned long long ctx = context_id();
    if (ctx == 0 || wi.ctx != ctx) {
        // Function attributes belong to the context: set them again in a new one.  The
        // limit is the device's; each split checks its own footprint against it.
        wi.ok = cudaFuncSetAttribute(hc_pre_wide_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     di.max_smem_optin) == cudaSuccess;
        if (!wi.ok)
            cudaGetLastError();
        wi.ctx = context_id();
    }
    return wi.ok;
}

struct WideWs {
    unsigned *pcount, *tcount, *flags;   // contiguous, zeroed by the launcher
    size_t counter_bytes;
    float *part, *red;
};

// Workspace layout after the 256-byte status block (and, in a phase-stamp build, the
// stamps): the tiles' counters and flags (zeroed by the launcher before each launch),
// the per-CTA partial slots (sized for up to kWMaxCtas CTAs) and the tiles' sums.
size_t wide_layout(int T, int s, char *base, WideWs *out)
{
    const int R = (2 + s) * s;
    const size_t ntiles = (size_t)(T + kWM - 1) / kWM;
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t o_ctr = kStatusBytes + kWorkspaceExtra;   // a phase-stamp build keeps its stamps first
    const size_t ctr_bytes = 3 * ntiles * 4;
    const size_t o_part = up(o_ctr + ctr_bytes);
    const size_t o_red = up(o_part + (size_t)kWNst * kWMaxCtas * kWM * (R + 1) * 4);
    const size_t o = up(o_red + (size_t)kWNst * kWM * (R + 1) * 4);
    if (out) {
        out->pcount = reinterpret_cast<unsigned *>(base + o_ctr);
        out->tcount = out->pcount + ntiles;
        out->flags = out->tcount + ntiles;
        out->counter_bytes = ctr_bytes;
        out->part = reinterpret_cast<float *>(base + o_part);
        out->red = reinterpret_cast<float *>(base + o_red);
    }
    return o;
}

template <int S>
cudaError_t run_wide(const float *x, const float *fn_w, const float *scale, const float *base, int T, int d,
                     int iters, float eps, float *pre, float *post, float *comb, float *y, void *workspace,
                     cudaStream_t st, const DeviceInfo &di)
{
    WideSplit sp;
    if (!wide_split(S, d, di, sp) || !wide_ready<S>(di))
        return cudaErrorNotSupported;
    WParams p = {};
    WideWs ws;
    wide_layout(T, S, static_cast<char *>(workspace), &ws);
    p.scale = scale;
    p.base = base;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.status = static_cast<StatusBlock *>(workspace);
    p.pcount = ws.pcount;
    p.tcount = ws.tcount;
    p.flags = ws.flags;
    p.part = ws.part;
    p.red = ws.red;
    p.T = T;
    p.d = d;
    p.ntiles = (T + kWM - 1) / kWM;
    p.ncta = sp.ncta;
    p.iters = iters;
    p.nwide = sp.nwide;
    p.hw0 = sp.hw0;
    p.hw1 = sp.hw1;
    p.eps = eps;
    p.invK = 1.0f / (float)(S * d);
#ifdef HC_STAMPS
    p.stamps = reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + kStatusBytes);
#endif
    constexpr int R = WG<S>::R;
    if (!w_encode(&p.tmap_x[0], x, T, S, d, sp.hw0, kWM) || !w_encode(&p.tmap_x[1], x, T, S, d, sp.hw1, kWM) ||
        !w_encode(&p.tmap_w[0], fn_w, R, S, d, sp.hw0, R) || !w_encode(&p.tmap_w[1], fn_w, R, S, d, sp.hw1, R))
        return cudaErrorInvalidValue;
    // The counters and flags start at zero whatever an earlier call left in the workspace.
    const cudaError_t e = cudaMemsetAsync(ws.pcount, 0, ws.counter_bytes, st);
    if (e != cudaSuccess)
        return e;
    const WLay L = make_wlay<S>(S * sp.hw0);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;   // every CTA resident at once: they poll each other's flags
    at[0].val.cooperative = 1;
    cfg.gridDim = dim3((unsigned)sp.ncta);
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hc_pre_wide_kernel<S>, p);
}

}  // namespace

size_t wide_workspace_bytes(int T, int s, int d)
{
    (void)d;
    if (s < 5 || s > 8)
        return kStatusBytes;
    return wide_layout(T, s, nullptr, nullptr);
}

bool wide_supported(int s, int d)
{
    DeviceInfo di;
    if (s < 5 || s > 8 || d % 4 != 0 || !device_info(di) || di.cc_major != 10)
        return false;
    WideSplit sp;
    if (!wide_split(s, d, di, sp))
        return false;
    switch (s) {
    case 5: return wide_ready<5>(di);
    case 6: return wide_ready<6>(di);
    case 7: return wide_ready<7>(di);
    case 8: return wide_ready<8>(di);
    default: return false;
    }
}

cudaError_t launch_pre_wide(const float *x, const float *fn_w, const float *scale, const float *base, int T, int s,
                            int d, int iters, float eps, float *pre, float *post, float *comb, float *y,
                            void *workspace, cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    switch (s) {
    case 5: return run_wide<5>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di);
    case 6: return run_wide<6>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di);
    case 7: return run_wide<7>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di);
    case 8: return run_wide<8>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace hc
