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
//    ring of shared-memory stages (the dot ring; a tile's slice is only a few KiB).
//  * Eight compute warps: warp w owns the w-th eighth of the LK columns; its lane
//    pair p (lanes 2p, 2p+1) owns rows [RB*p, RB*p+RB) (RB = ceil(R/16)), each lane
//    of the pair one half of the warp's columns, and every lane does all kWM tokens
//    of a tile.  Packed float32 FMAs (x from shared memory, four columns a step;
//    fn_w from TMEM, the next step's load in flight); the pair's halves are added by
//    one shuffle level and each warp leaves its values in one of kWNb shared-memory
//    buffers, then goes on with the next tile: a compute warp waits for the others
//    only when it is kWNb tiles ahead of the slowest.
//  * A publisher warp, once the eight warps have left a tile's values, refills the
//    stage the tile used, sums the eight warps' values in warp order into the tile's
//    partial dots and sums of squares (a slot of the workspace), frees the buffer and
//    raises the tile's counter.
//  * Tiles are finished by fixed, rotating CTAs (no CTA's share of the work depends
//    on its timing), in two steps: each of the 4*RV/4 float4 columns of a tile's
//    partial rows has a reducer CTA, which sums that column over every CTA's row
//    (lanes over rows, then a fixed xor tree: one round trip to L2); the tile's
//    finisher gathers the reduced columns, forms the gates (pre and post written
//    out), sets the tile's flag and then runs the tile's Sinkhorn.  Each CTA has one
//    warp for each step; each takes its duties in tile order and waits (bounded) for
//    the counters they need.
//  * A collapse warp in every CTA takes the runs of tiles whose flags are set (a
//    bounded wait for the first), loads their gates in one round trip and writes y for
//    the CTA's hidden columns from its own ring (the collapse ring), which loads the
//    tile's slice a second time, some tens of microseconds after the dot ring did: the
//    dot ring's loads keep the lines in L2 (evict_last) and no CTA runs more than kWNp
//    tiles ahead, so x comes from HBM about once.  The dot ring never waits for a
//    tile's cross-CTA chain; it waits only for the partial slot it writes to, kWNp
//    tiles on.  No wait depends on a later tile, so the grid cannot deadlock.
//  * Every wait is bounded (2 s); on timeout the kernel records the site in the
//    workspace status word and winds down.  The host zeroes the tiles' counters and
//    flags (a memset on the stream) before each launch, so what other paths or
//    earlier calls left in the workspace does not matter.
//
// Determinism: every partial has a fixed summation order (per lane in column order,
// the lane pair's halves, the eight warps in warp order), the partials of a token are
// summed over CTAs in a fixed order (per lane over CTAs l, l+32, ..., then an xor
// tree), and no float atomics are used: repeated calls give the same bits, and a
// token's results do not depend on the other tokens of the batch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>

#include "hc_internal.cuh"
#include "hc_ptx.cuh"

namespace hc {
namespace {

constexpr int kWThreads = 384;            // 12 warps
constexpr int kWNCW = 8;                  // compute warps 0-7, one eighth of the slice each
constexpr int kWPublishWarp = 8;          // publishes this CTA's partials, refills the dot ring
constexpr int kWReduceWarp = 9;           // column sums of the (tile, column) pairs this CTA reduces
constexpr int kWTileWarp = 10;            // tile finishes (gates, flag, Sinkhorn) of this CTA's tiles
constexpr int kWCollapseWarp = 11;        // collapse, with its own ring
constexpr int kWM = 4;                    // tokens per tile
constexpr int kWNstMax = 16;              // dot-ring stages (the launcher fits as many as it can)
constexpr int kWNcsMax = 8;               // collapse-ring stages
constexpr int kWNp = 64;                  // partial and tile-sum slots in the workspace (bounds how far a CTA runs ahead)
constexpr int kWNb = 4;                   // buffers of the compute warps' values
constexpr int kWMaxCtas = 160;            // workspace sizing bound on the grid
constexpr uint32_t kWTmemCols = 256;
constexpr int kWMaxTmemCols = 256;
constexpr unsigned long long kWWaitNs = 2000000000ull;
constexpr unsigned kFullMask = 0xffffffffu;

enum WSite : unsigned {
    kWSiteW = 32, kWSiteFull, kWSiteLeft, kWSiteFlag, kWSiteReduce, kWSiteTile, kWSiteDrain, kWSiteSlot, kWSiteCFull,
    kWSiteFreed
};

template <int S>
struct WG {
    static constexpr int R = (2 + S) * S;
    static constexpr int RB = (R + 15) / 16;                // rows per lane pair
    static constexpr int WB = 4 * RB;                        // TMEM columns per four-column step
    static constexpr int RP = 16 * RB;                       // rows padded to the 16 lane pairs
    static constexpr int RS = RP + 4;                        // token stride of the cross-warp area
    static constexpr int RV = R + 1;                         // partial values per token: R dots + sum of squares
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
    float *part;        // [kWNp][ncta][kWM][RV]: each CTA's partials of a tile
    float *red;         // [kWNp][kWM][RV]: the tile's sums over every CTA
    int T, d, ntiles, ncta, iters;
    int y_rows;            // rows of y (T): bounds of the bounds-checked build's y stores
    int nst, ncs;          // dot-ring and collapse-ring stages
    int nwide, hw0, hw1;   // CTAs [0, nwide) own hw0 columns, the rest hw1
    float eps, invK;       // invK = 1 / (s*d)
    unsigned long long *stamps;   // phase stamps (HC_STAMPS builds), else null
};

// Phase stamps (HC_STAMPS builds only).  Slot 0: CTA 0's compute warp 0
// (kEvStageReady, kEvDotsDone, kEvShipped), publisher (kEvPartials; kEvRefilled at
// tile k when it loads tile k + nst) and collapse warp (kEvPreArrived, kEvCollapsed).  Slot 1, whichever CTA does it: the
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
    int stage_bytes, off_cst, off_scr, off_red, off_ex, off_bar, off_misc, total;
};

// Shared memory: the dot ring [nst] and the collapse ring [ncs] of stages (together
// with the cross-warp area they also hold the fn_w slice while it is copied to TMEM),
// the compute warps' cross-warp area, the finisher's tile sums and exps, the collapse
// warp's gates, the barriers and a few words.
template <int S>
__host__ __device__ inline WLay make_wlay(int lk_max, int nst, int ncs)
{
    using G = WG<S>;
    WLay L;
    L.stage_bytes = kWM * lk_max * 4;
    int o = nst * L.stage_bytes;
    L.off_cst = o;
    o += ncs * L.stage_bytes;
    L.off_scr = o;                   // [kWNb][kWNCW][kWM][RS]: the compute warps' values of kWNb tiles
    o += kWNb * kWNCW * kWM * G::RS * 4;
    L.off_red = o;                   // [kWM][RV]: the finished tile's summed partials
    o += kWM * G::RV * 4;
    o = (o + 15) / 16 * 16;
    L.off_ex = o;                    // [kWM][S*S]: the finished tile's exp(comb logits),
    o += kWM * S * S * 4;            // then [kWNcsMax][kWM][S]: the collapse warp's copy of the
    o += kWNcsMax * kWM * S * 4;     // pre gates of the tiles it is collapsing
    o = (o + 7) / 8 * 8;
    L.off_bar = o;                   // full[kWNstMax], cfull[kWNcsMax], wfull, left[kWNb], freed[kWNb]
    o += (kWNstMax + kWNcsMax + 1 + 2 * kWNb) * 8;
    L.off_misc = o;                  // TMEM address, abort flag, TMA loads issued per stage
    o += 16 + (kWNstMax + kWNcsMax) * 4;
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

// One level of an xor reduce-scatter over the lanes of a warp: lanes whose M bit is clear
// keep the lower half of the list and add their partner's copy of it, the others the
// upper half (used with M = 1 for a lane pair's halves and M = 4, 2, 1 for the
// Sinkhorn's column sums over a token's eight lanes).
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
template <int N>
__device__ __forceinline__ float w_tree_sum(const float *v)
{
    if constexpr (N == 1) {
        return v[0];
    } else {
        return w_tree_sum<N / 2>(v) + w_tree_sum<N - N / 2>(v + N / 2);
    }
}

// Sinkhorn of the tile's kWM matrices, one row per lane: lane (t, j) = (lane >> 3,
// lane & 7) holds row j of token t's S x S matrix (rows j >= S and tokens t >= tm are
// zeros).  Each of `iters` rounds divides every row by (row sum + eps), then every
// column by (column sum + eps), with correctly rounded reciprocals; a column's sum
// comes from a three-level xor reduce-scatter over the token's eight lanes (lane j
// ends with column j) and its reciprocal is passed round by shuffles.
template <int S>
__device__ __forceinline__ void w_sinkhorn_rows(float *c, int iters, float eps, int lane)
{
    static_assert(S <= 8, "one lane per row, eight lanes per token");
    for (int it = 0; it < iters; ++it) {
        const float rinv = 1.0f / (w_tree_sum<S>(c) + eps);
#pragma unroll
        for (int k = 0; k < S; ++k)
            c[k] *= rinv;
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            v[k] = k < S ? c[k] : 0.f;
        w_rs_level<8, 4>(v, lane);
        w_rs_level<4, 2>(v, lane);
        w_rs_level<2, 1>(v, lane);
        const float cinv = 1.0f / (v[0] + eps);
#pragma unroll
        for (int k = 0; k < S; ++k)
            c[k] *= __shfl_sync(kFullMask, cinv, (lane & ~7) | k);
    }
}

template <int S>
__global__ void __launch_bounds__(kWThreads, 1) hc_pre_wide_kernel(const __grid_constant__ WParams p)
{
    using G = WG<S>;
    constexpr int R = G::R, RB = G::RB, WB = G::WB, RP = G::RP, RS = G::RS, RV = G::RV;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const int hw = cta < p.nwide ? p.hw0 : p.hw1;
    const int h0 = cta < p.nwide ? cta * p.hw0 : p.nwide * p.hw0 + (cta - p.nwide) * p.hw1;
    const int LK = S * hw;
    const int nst = p.nst, ncs = p.ncs;
    const WLay L = make_wlay<S>(S * p.hw0, nst, ncs);
    const CUtensorMap *tmx = &p.tmap_x[cta < p.nwide ? 0 : 1];
    const CUtensorMap *tmw = &p.tmap_w[cta < p.nwide ? 0 : 1];
    float *stages = reinterpret_cast<float *>(smem);
    float *cstages = reinterpret_cast<float *>(smem + L.off_cst);
    float *scr = reinterpret_cast<float *>(smem + L.off_scr);
    float *red = reinterpret_cast<float *>(smem + L.off_red);
    float *ex = reinterpret_cast<float *>(smem + L.off_ex);
    const uint32_t bar0 = ptx::smem_u32(smem + L.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L.off_misc + 16);   // per dot stage
    volatile int *cissued = issued + kWNstMax;                                          // per collapse stage
    StatusBlock *sb = p.status;
    const int stage_floats = L.stage_bytes / 4;
    auto FULL = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto CFULL = [&](int s) { return bar0 + 8u * (uint32_t)(kWNstMax + s); };
    const uint32_t WFULL = bar0 + 8u * (uint32_t)(kWNstMax + kWNcsMax);
    // LEFT(b): the eight compute warps have left a tile's values in buffer b (and are
    // done with its stage); FREED(b): the publisher has summed them.
    auto LEFT = [&](int b) { return bar0 + 8u * (uint32_t)(kWNstMax + kWNcsMax + 1 + b); };
    auto FREED = [&](int b) { return bar0 + 8u * (uint32_t)(kWNstMax + kWNcsMax + 1 + kWNb + b); };
    const uint32_t tile_bytes = (uint32_t)(kWM * LK * 4);
    // The dot ring's loads keep the tile's lines in L2 (evict_last) for the collapse ring,
    // which reads the same slice again a few tens of microseconds later, for the last time
    // (evict_first): x then comes from HBM once.
    auto load_tile = [&](int it) {   // one thread; the dot stage must be free
        const int s = it % nst;
        ptx::mbar_arrive_expect_tx(FULL(s), tile_bytes);
        ptx::tma_load_3d_hint(ptx::smem_u32(stages + s * stage_floats), tmx, h0, 0, it * kWM, FULL(s),
                              ptx::l2_evict_last());
        issued[s] = issued[s] + 1;
    };
    auto load_ctile = [&](int it) {   // one thread; the collapse stage must be free
        const int s = it % ncs;
        ptx::mbar_arrive_expect_tx(CFULL(s), tile_bytes);
        ptx::tma_load_3d_hint(ptx::smem_u32(cstages + s * stage_floats), tmx, h0, 0, it * kWM, CFULL(s),
                              ptx::l2_evict_first());
        cissued[s] = cissued[s] + 1;
    };

    // ------------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        W_STAMP(0, kEvKernelStart);
        for (int s = 0; s < kWNstMax; ++s) {
            ptx::mbar_init(FULL(s), 1);
            issued[s] = 0;
        }
        for (int b = 0; b < kWNb; ++b) {
            ptx::mbar_init(LEFT(b), kWNCW);   // every compute warp arrives once per tile
            ptx::mbar_init(FREED(b), 1);
        }
        for (int s = 0; s < kWNcsMax; ++s) {
            ptx::mbar_init(CFULL(s), 1);
            cissued[s] = 0;
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

    // This CTA's fn_w slice, staged through shared memory, to the compute warps' TMEM
    // lanes: step q (four columns) at columns q*WB .., row r of the lane's pair at
    // 4r .. 4r+3 (rows past R are zeros).
    const int sp = warp & 3;
    const int rg = lane >> 1, kh = lane & 1;                  // lane pair (row group) and column half
    const int KH = LK / 16, NQS = KH / 4;                     // columns per lane; four-column steps
    const int kbase = warp * (LK / 8) + kh * KH;              // the lane's first column of the slice
    const uint32_t trow = tmem_base + ((uint32_t)(32 * sp) << 16) + (uint32_t)((warp >> 2) * WB * NQS);
    bool ok = !skip;
    if (ok && threadIdx.x == 0) {
        ptx::prefetch_tmap(tmx);
        ptx::prefetch_tmap(tmw);
        ptx::mbar_arrive_expect_tx(WFULL, (uint32_t)(R * LK * 4));
        ptx::tma_load_3d(ptx::smem_u32(stages), tmw, h0, 0, 0, WFULL);
    }
    if (ok && warp < kWNCW) {
        ok = w_warp_wait(lane, WFULL, 0, abort_flag, sb, kWSiteW);
        if (ok) {
            const float *wst = stages;
            for (int q = 0; q < NQS; ++q) {
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int row = rg * RB + r;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row < R)
                        v = *reinterpret_cast<const float4 *>(wst + row * LK + kbase + 4 * q);
                    const float a[4] = {v.x, v.y, v.z, v.w};
                    ptx::tmem_st4(trow + (uint32_t)(q * WB + 4 * r), a);
                }
            }
            ptx::tmem_wait_st();
        }
    }
    ptx::tmem_fence_before_sync();
    ok = __syncthreads_and(ok ? 1 : 0) != 0;   // the staged slice may be overwritten now
    ptx::tmem_fence_after_sync();

    if (ok && warp < kWNCW) {
        // -------------------------------------------------------------- compute warps
        if (threadIdx.x == 0)
            for (int it = 0; it < nst && it < p.ntiles; ++it)
                load_tile(it);
        // The lane's sum-of-squares token: pair p < kWM sums token p (both halves).
        const uint32_t sq_off = 4u * (uint32_t)((rg & 3) * LK);
        for (int it = 0; it < p.ntiles; ++it) {
            const int s = it % nst;
            if (!w_warp_wait(lane, FULL(s), (it / nst) & 1, abort_flag, sb, kWSiteFull))
                break;
            if (threadIdx.x == 0)
                W_STAMP(it, kEvStageReady);
            const uint32_t xs = ptx::smem_u32(stages + s * stage_floats) + 4u * (uint32_t)kbase;
            float2 acc[kWM][RB];
            float2 ssa = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kWM; ++i)
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    acc[i][r] = make_float2(0.f, 0.f);
            float wa[WB], wb[WB];
            ptx::tmem_ld_issue<WB>(trow, wa);
            ptx::tmem_ld_wait_regs<WB>(wa);
            // One four-column step with fn_w values wc; the next step's values are loaded
            // into wn meanwhile.
            auto step = [&](int q, float *wc, float *wn) {
                const bool more = q + 1 < NQS;
                if (more)
                    ptx::tmem_ld_issue<WB>(trow + (uint32_t)((q + 1) * WB), wn);
                float4 xv[kWM];
#pragma unroll
                for (int i = 0; i < kWM; ++i)
                    xv[i] = ptx::lds128(xs + (uint32_t)(i * LK * 4 + q * 16));
                const float4 xq = ptx::lds128(xs + sq_off + (uint32_t)(q * 16));
#pragma unroll
                for (int i = 0; i < kWM; ++i)
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        acc[i][r] = ptx::ffma2(make_float2(xv[i].x, xv[i].y), make_float2(wc[4 * r], wc[4 * r + 1]),
                                               acc[i][r]);
                        acc[i][r] = ptx::ffma2(make_float2(xv[i].z, xv[i].w),
                                               make_float2(wc[4 * r + 2], wc[4 * r + 3]), acc[i][r]);
                    }
                ssa = ptx::ffma2(make_float2(xq.x, xq.y), make_float2(xq.x, xq.y), ssa);
                ssa = ptx::ffma2(make_float2(xq.z, xq.w), make_float2(xq.z, xq.w), ssa);
                if (more)
                    ptx::tmem_ld_wait_regs<WB>(wn);
            };
            int q = 0;
            for (; q + 1 < NQS; q += 2) {
                step(q, wa, wb);
                step(q + 1, wb, wa);
            }
            if (q < NQS)
                step(q, wa, wb);
            if (threadIdx.x == 0)
                W_STAMP(it, kEvDotsDone);
            // The lane pair's halves: lane kh keeps tokens 2kh, 2kh+1 of its rows.
            float v[kWM * RB];
#pragma unroll
            for (int i = 0; i < kWM; ++i)
#pragma unroll
                for (int r = 0; r < RB; ++r)
                    v[i * RB + r] = acc[i][r].x + acc[i][r].y;
            w_rs_level<kWM * RB, 1>(v, lane);
            float sq = ssa.x + ssa.y;
            sq += __shfl_xor_sync(kFullMask, sq, 1);
            // This warp's values -> buffer it % kWNb, once the publisher has summed the
            // tile kWNb earlier: [warp][token][row], the sum of squares of token t at
            // row RP.
            const int b = it % kWNb;
            if (it >= kWNb && !w_warp_wait(lane, FREED(b), ((it / kWNb) - 1) & 1, abort_flag, sb, kWSiteFreed))
                break;
            float *area = scr + ((size_t)b * kWNCW + warp) * kWM * RS;
#pragma unroll
            for (int m = 0; m < 2 * RB; ++m) {
                const int i = 2 * kh + m / RB, row = rg * RB + (m - (m / RB) * RB);
                area[i * RS + row] = v[m];
            }
            if (kh == 0 && rg < kWM)
                area[rg * RS + RP] = sq;
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(LEFT(b));   // release: the values, and the stage is done with
            if (threadIdx.x == 0)
                W_STAMP(it, kEvShipped);
        }
    } else if (ok && warp == kWPublishWarp) {
        // -------------------------------------------------------------- publisher warp
        // Tile by tile, once the eight compute warps have left its values: refill the
        // stage with the tile nst on, sum the eight warps' values in warp order (into
        // registers, then the buffer is freed), and store them to the tile's partial
        // slot.  A refill for tile nx first makes sure that the flag of tile nx - kWNp
        // is set (its partial and tile-sum slots are reused): flags are read 32 at a
        // time and the run of set ones remembered, with a bounded wait when none is.
        // The tiles' counters are raised in runs: one fence for every tile summed so
        // far, as soon as the next tile's values are not already waiting.
        constexpr int NO = (kWM * RV + 31) / 32;   // outputs per lane
        int gchk = 0;       // flags [0, gchk) are known to be set
        int pend = 0;       // tiles [pend, it] are stored but their counters not raised
        for (int it = 0; it < p.ntiles; ++it) {
            const int b = it % kWNb;
            if (!w_warp_wait(lane, LEFT(b), (it / kWNb) & 1, abort_flag, sb, kWSiteLeft))
                break;
            bool good = true;
            if (it + nst < p.ntiles) {
                const int nx = it + nst;
                while (nx - kWNp >= gchk) {
                    const unsigned f = gchk + lane < p.ntiles ? ptx::ld_acquire_gpu(&p.flags[gchk + lane]) : 0u;
                    const unsigned run = __ballot_sync(kFullMask, f != 0u);
                    if (run == kFullMask)
                        gchk += 32;
                    else if (run & 1u)
                        gchk += __ffs(~run) - 1;
                    else if (!(good = w_warp_wait_count(lane, &p.flags[gchk], 1u, abort_flag, sb, kWSiteSlot)))
                        break;
                }
                if (!good)
                    break;
                if (lane == 0) {
                    load_tile(nx);
                    W_STAMP(it, kEvRefilled);
                }
            }
            const float *areas = scr + (size_t)b * kWNCW * kWM * RS;
            float sums[NO];
#pragma unroll
            for (int j = 0; j < NO; ++j) {
                const int o = lane + 32 * j;
                sums[j] = 0.f;
                if (o < kWM * RV) {
                    const int i = o / RV, r = o - (o / RV) * RV;
                    const int col = i * RS + (r < R ? r : RP);
                    float a = areas[col];
#pragma unroll
                    for (int w2 = 1; w2 < kWNCW; ++w2)
                        a += areas[w2 * kWM * RS + col];
                    sums[j] = a;
                }
            }
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(FREED(b));
            float *dst = p.part + ((size_t)(it % kWNp) * p.ncta + cta) * kWM * RV;
#pragma unroll
            for (int j = 0; j < NO; ++j) {
                const int o = lane + 32 * j;
                if (o < kWM * RV)
                    dst[o] = sums[j];
            }
            bool later = it + 1 < p.ntiles && it + 1 - pend < 8;
            if (later && lane == 0)
                later = ptx::mbar_test_wait(LEFT((it + 1) % kWNb), ((it + 1) / kWNb) & 1);
            if (!__shfl_sync(kFullMask, later, 0)) {
                __syncwarp();
                if (lane == 0) {
                    __threadfence();   // every lane's stores of the run, before the counters
                    for (int k = pend; k <= it; ++k) {
                        atomicAdd(&p.pcount[k], 1u);
                        W_STAMP(k, kEvPartials);
                    }
                }
                pend = it + 1;
            }
            __syncwarp();
        }
    } else if (ok && warp == kWReduceWarp) {
        // -------------------------------------------------------------- reduce warp
        // The column sums of the (tile, column) pairs this CTA reduces: column q of tile
        // it goes to CTA (it*Q4 + q) % ncta; duties in order of it, then q.
        constexpr int Q4 = kWM * RV / 4;
        static_assert((kWM * RV) % 4 == 0, "partial rows are whole float4s");
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
            const int slot = it % kWNp;
            const float4 *src = reinterpret_cast<const float4 *>(p.part + (size_t)slot * p.ncta * kWM * RV);
            float4 *dst = reinterpret_cast<float4 *>(p.red + (size_t)slot * kWM * RV);
            int nq = 0;
            for (; q < Q4; q += p.ncta, ++nq) {
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
                atomicAdd(&p.tcount[it], (unsigned)nq);
                if (cta == base)
                    W_STAMP_ANY(it, kEvXfDone);
            }
            __syncwarp();
        }
    } else if (ok && warp == kWTileWarp) {
        // -------------------------------------------------------------- tile warp
        // The finish of the tiles this CTA owns (tile it to CTA it % ncta): gather the
        // column sums, form the gates, set the flag, then the Sinkhorn.
        constexpr int Q4 = kWM * RV / 4;
        for (int it = cta; it < p.ntiles; it += p.ncta) {
            if (!w_warp_wait_count(lane, &p.tcount[it], (unsigned)Q4, abort_flag, sb, kWSiteTile))
                break;
            if (lane == 0)
                W_STAMP_ANY(it, kEvXfLanded);
            const float4 *src = reinterpret_cast<const float4 *>(p.red + (size_t)(it % kWNp) * kWM * RV);
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
                        store_checked(p.pre, (size_t)(t0 + i) * S + r, (size_t)p.T * S, sg + p.eps, p.status, kStorePre);
                    else
                        store_checked(p.post, (size_t)(t0 + i) * S + (r - S), (size_t)p.T * S, 2.f * sg, p.status,
                                      kStorePost);
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
            // The tile's Sinkhorn, one row per lane (this warp's next tile is ncta tiles on).
            const int t = lane >> 3, j = lane & 7;
            const bool act = t < tm && j < S;
            float cm[S];
#pragma unroll
            for (int k = 0; k < S; ++k)
                cm[k] = act ? ex[t * S * S + j * S + k] : 0.f;
            w_sinkhorn_rows<S>(cm, p.iters, p.eps, lane);
            if (act) {
#pragma unroll
                for (int k = 0; k < S; ++k)
                    store_checked(p.comb, (size_t)(t0 + t) * S * S + j * S + k, (size_t)p.T * S * S, cm[k], p.status,
                                  kStoreComb);
            }
            __syncwarp();
            if (lane == 0)
                W_STAMP_ANY(it, kEvSinkDone);
        }
    } else if (ok && warp == kWCollapseWarp) {
        // -------------------------------------------------------------- collapse warp
        // In runs of tiles: wait for the flag of the next tile, take the run of tiles
        // whose flags are already set (at most ncs), load their pre gates at once, then
        // tile by tile write y for this CTA's hidden columns from the collapse ring and
        // refill that stage with the tile ncs on.
        const int h4n = hw / 4;
        float *pre_s = ex + kWM * S * S;   // [kWNcsMax][kWM][S]: the gates of the run
        if (lane == 0)
            for (int it = 0; it < ncs && it < p.ntiles; ++it)
                load_ctile(it);
        __syncwarp();
        int it = 0;
        bool good = true;
        while (good && it < p.ntiles) {
            if (!w_warp_wait_count(lane, &p.flags[it], 1u, abort_flag, sb, kWSiteFlag))
                break;
            const int nmax = min(ncs, p.ntiles - it);
            const unsigned f = lane < nmax ? ptx::ld_acquire_gpu(&p.flags[it + lane]) : 0u;
            const unsigned run = __ballot_sync(kFullMask, f != 0u) | 1u;   // tile it's flag is set
            const int n = min(nmax, __ffs(~run) - 1);
            __threadfence();   // every lane reads gates that other lanes' flags cover
            const int t0 = it * kWM, ntok = min(n * kWM, p.T - t0);
            for (int e = lane; e < ntok * S; e += 32)
                pre_s[e] = __ldcg(p.pre + (size_t)t0 * S + e);
            __syncwarp();
            for (int b = 0; b < n; ++b, ++it) {
                if (lane == 0)
                    W_STAMP(it, kEvPreArrived);
                const int s = it % ncs;
                if (!(good = w_warp_wait(lane, CFULL(s), (it / ncs) & 1, abort_flag, sb, kWSiteCFull)))
                    break;
                const int tm = min(kWM, p.T - it * kWM);
                const float *xs = cstages + s * stage_floats;
                for (int e = lane; e < tm * h4n; e += 32) {
                    const int i = e / h4n, c4 = e - (e / h4n) * h4n;
                    const float *pr = pre_s + (b * kWM + i) * S;
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
                    store_checked(reinterpret_cast<float4 *>(p.y), ((size_t)(it * kWM + i) * p.d + h0 + 4 * c4) / 4,
                                  (size_t)p.y_rows * p.d / 4, a, p.status, kStoreY);
                }
                __syncwarp();
                if (lane == 0) {
                    W_STAMP(it, kEvCollapsed);
                    if (it + ncs < p.ntiles)
                        load_ctile(it + ncs);
                }
                __syncwarp();
            }
            __syncwarp();   // the run's gates are free
        }
    }

    // ------------------------------------------------------------------ teardown
    ptx::tmem_fence_before_sync();
    __syncthreads();
    if (threadIdx.x == 0) {
        // Every TMA load this CTA issued lands before it exits.
        if (!skip)
            w_wait_bar(WFULL, 0, abort_flag, sb, kWSiteDrain, false);
        for (int s = 0; s < kWNstMax; ++s)
            if (issued[s] > 0)
                w_wait_bar(FULL(s), (issued[s] - 1) & 1, abort_flag, sb, kWSiteDrain, false);
        for (int s = 0; s < kWNcsMax; ++s)
            if (cissued[s] > 0)
                w_wait_bar(CFULL(s), (cissued[s] - 1) & 1, abort_flag, sb, kWSiteDrain, false);
    }
    __syncthreads();
    ptx::tmem_fence_after_sync();
    if (warp == 0)
        ptx::tmem_dealloc(tmem_base, kWTmemCols);
}

// ---------------------------------------------------------------------- host side

// Map a row-major [rows][s][d] float tensor as (d, s, rows) with a box (hw, s, box_rows);
// reads past the last row are zero-filled.
bool w_encode(CUtensorMap *m, const float *base, int rows, int s, int d, int hw, int box_rows)
{
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)s, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 4, (cuuint64_t)s * d * 4};   // bytes
    const cuuint32_t box[3] = {(cuuint32_t)hw, (cuuint32_t)s, (cuuint32_t)box_rows};
    return tensor_map_f32(m, 3, base, dims, strides, box);
}

// The hidden split: widths are multiples of the unit u (the smallest multiple of 8 with
// s*u % 64 == 0), at most one unit apart, over as many CTAs as the device has SMs.
struct WideSplit {
    int ncta = 0, nwide = 0, hw0 = 0, hw1 = 0;
    int nst = 0, ncs = 0;   // dot-ring and collapse-ring stages that fit
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
    if (lk_max % 64 != 0 || 2 * G::WB * (lk_max / 64) > kWMaxTmemCols)   // two compute warps share each TMEM lane
        return false;
    // As many dot-ring stages as fit (at least 4), then collapse-ring stages (at least 2).
    int nst = kWNstMax, ncs = kWNcsMax;
    while (nst > 4 && make_wlay<S>(lk_max, nst, ncs).total > max_smem)
        --nst;
    while (ncs > 2 && make_wlay<S>(lk_max, nst, ncs).total > max_smem)
        --ncs;
    const WLay L = make_wlay<S>(lk_max, nst, ncs);
    if (L.total > max_smem)
        return false;
    if (G::R * lk_max * 4 > L.off_red)   // the fn_w slice is staged through the rings and value buffers
        return false;
    w.nst = nst;
    w.ncs = ncs;
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
    const size_t o_red = up(o_part + (size_t)kWNp * kWMaxCtas * kWM * (R + 1) * 4);
    const size_t o = up(o_red + (size_t)kWNp * kWM * (R + 1) * 4);
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
    p.nst = sp.nst;
    p.ncs = sp.ncs;
    p.eps = eps;
    p.invK = 1.0f / (float)(S * d);
    p.y_rows = T;
#ifdef HC_DEBUG_BOUNDS
    // Bounds-checked build only: pretend y has fewer rows, so that the checks' report can be
    // tested (the stores they refuse are inside the real buffer).
    if (const char *e = getenv("HC_DEBUG_BOUNDS_Y_ROWS"))
        p.y_rows = atoi(e);
#endif
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
    const WLay L = make_wlay<S>(S * sp.hw0, sp.nst, sp.ncs);
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
