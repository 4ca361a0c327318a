// hc_pre_cluster.cu -- the fused pre-chain: one launch per site, x read from HBM once.
//
// What it computes (memra-engine hyper.rs page, module header "ARITHMETIC
// CONTRACT"): per token, mixes = fn_w . x[t] over the whole s*d slab, rescaled
// by rsqrt(mean(x[t]^2) + eps); the pre/post gates and the Sinkhorn comb from
// the logits mixes*scale[group] + base; the collapse y[t] = sum_c pre_c x[t,c].
//
// How (GB300 design):
//  * A thread-block cluster of kCS = 16 CTAs splits the hidden dimension: CTA c
//    owns hidden columns [c*hs, (c+1)*hs), hs = d/16, of every stream, i.e. an
//    LK = s*hs column slice of each token's slab and the matching LK columns
//    of all R rows of fn_w.  Because the slice covers all s streams of its
//    hidden range, the collapse of that range needs nothing from other CTAs.
//  * Each token tile (<= 16 tokens) arrives by one tiled TMA load (a 4-D tensor
//    map whose box is the CTA's column slice of every stream of the tile's
//    tokens) into a shared-memory stage and stays there until its collapse, so
//    x is read from HBM exactly once.
//  * The fn_w slice (one more TMA box) stays resident in the CTA for every tile
//    it processes: in tensor memory (TMEM, tcgen05.ld into registers) for the
//    persistent prefill variant, in shared memory for the one-tile decode
//    variant.  It is read from L2/HBM once per CTA.
//  * Eight compute warps run the contraction.  Persistent variant: warp w owns
//    rows [B*(w&1), B*(w&1)+B) (B = 12 for s = 4), column half (w>>1)&1 and
//    token slots [8*(w/4), 8*(w/4)+8), so every x value of a stage is read by
//    two warps; decode variant: rows [B*(w%4), ..) (B = 6), column half w/4,
//    every token slot.  In a warp, lanes 0-15 take the first of its token slots
//    and lanes 16-31 the rest, and lane&15 is the K-group kg owning columns
//    2kg, 2kg+1, 32+2kg, 33+2kg of every 64-column group (so each half-warp
//    load is 128 contiguous bytes).  Operands: x from shared memory, fn_w from TMEM; packed
//    float32 FMAs on CUDA cores (no TF32: the 24-row contraction is too skinny
//    for tensor cores and must stay in f32).  A 16-lane xor reduce-scatter
//    sums the K-groups, and each lane stores its partial dots and sums of
//    squares straight into the owner CTA's receive buffer (token t of a tile
//    belongs to CTA t) with st.async, which counts the bytes on the owner's
//    mbarrier.  Then they go on to the next tile: they never wait for gates.
//  * Persistent variant: the two warpgroups of compute warps wait for tiles on
//    their own barriers, warpgroup 1 starting a tile later than warpgroup 0, so
//    one reduces and ships while the other runs its FMAs.  Four
//    collapse warps (one per SM sub-partition) wait for each tile's pre gates,
//    write y for the CTA's hidden columns from the tile's stage and refill the
//    stage, so the stage ring alone couples them to the compute warps.  In the
//    fused post -> pre mode they also apply the previous site's hc_post to each
//    landed tile in place (x -> x', two tiles ahead of their collapse), store x'
//    by TMA and release the stage to the compute warps.  The decode variant's
//    single tile is transformed and collapsed by the compute warps.  The
//    sixteen warps launch at 128 registers; the two compute warpgroups raise
//    theirs to 192 with setmaxnreg while the finisher warpgroup drops to 48 and
//    the collapse warpgroup to 80.
//  * Two finisher warps (even/odd tiles) of each owner sum the 2 x 16
//    partials in a fixed tree, apply the rsqrt rescale, form the gates,
//    broadcast pre to all 16 CTAs and write pre/post; exp(comb logits) go to
//    the tile's Sinkhorn CTA (tile index mod 16), whose Sinkhorn warp
//    normalises all the tile's comb blocks at once, one token per lane, in
//    registers, off the path that the next tiles' gates take.
//  * Branch-input norm mode (hc_pre_fused_norm): after a tile's collapse each CTA
//    sends its share of every token's sum of y^2 to the other fifteen (st.async,
//    an 8-slot exchange over the f buffer, which this mode does not use) and then
//    writes z = y * rsqrt(mean(y^2) + eps_norm) * norm_w and its Q8_0 pair for its
//    own columns (the persistent variant one tile later, from the sum it took
//    while writing y; the decode variant reads its tile back).
//  * Every wait on an mbarrier is bounded (2 s of %globaltimer); on timeout the
//    kernel records the site in the workspace status word, stops issuing work,
//    lets its TMA loads land, meets the other CTAs at the final cluster
//    barrier, frees TMEM and returns.  A launch that finds the status word
//    already set does nothing at all.
//
// Determinism: every sum has a fixed order independent of T, of the tile a
// token lands in and of the variant, so a token's outputs are the same bits
// whatever batch it is in.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hc_internal.cuh"
#include "hc_ptx.cuh"

#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <mutex>

namespace hc {
namespace {

constexpr int kCS = 16;              // CTAs per cluster (non-portable cluster size)
constexpr int kTMT = 16;             // max tokens per tile = one owner CTA per token
constexpr int kNCW = 8;              // compute warps: two per SM sub-partition
constexpr int kFinisherWarp = 8;     // warps 8 and 9 take even and odd tiles
constexpr int kSinkWarp = 10;        // the Sinkhorn of the tiles this CTA normalises
constexpr int kCollapseWarp0 = 12;   // persistent variant: warps 12-15 collapse tiles, refill stages
constexpr int kCollapseThreads = 4 * 32;
constexpr int kThreads = 16 * 32;    // four warpgroups, launched at 128 registers a thread
// The two compute warpgroups take registers from the other two (whose warps wait
// or stream shared memory): 2 x 128 x 192 + 128 x 48 (finisher / Sinkhorn warps)
// + 128 x 80 (collapse warps, which also run the fused mode's tile transform) = 512 x 128.  The split
// is made once, at the role dispatch, and kept until exit: a warpgroup that gave
// registers back and then asked for them again could take them before the compute
// warpgroups had theirs, and those would then wait for registers forever.
constexpr int kRegsCompute = 192, kRegsFinish = 48, kRegsCollapse = 80;
static_assert(2 * 128 * kRegsCompute + 128 * kRegsFinish + 128 * kRegsCollapse == kThreads * 128, "register split");
// Named barriers: 1 all compute warps, 2 collapse warps, 3 + g compute warpgroup g of the
// persistent variant (its tile barrier), 5 the warpgroups' one-off start stagger.
constexpr uint32_t kNbCompute = 1, kNbCollapse = 2, kNbGroup0 = 3, kNbStagger = 5;
constexpr int kSinkLag = 8;          // a finisher waits for the Sinkhorn of the tile 8 before its own
constexpr int kComputeThreads = kNCW * 32;
constexpr int kNstPersist = 3;
constexpr int kMaxLK = 1024;         // s*d/16 <= 1024: three 64 KiB stages fit in shared memory
constexpr int kMaxFusedHs = 256;     // fused post -> pre: f slice of <= 256 columns (16 KiB a tile)
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;

// mbarrier slots
// Exchange buffers rotate over kNQ tiles (tile it uses slot it % kNQ).  Bytes for
// tile it + 3 reach this CTA only after it has shipped tile it + 3, whose stage its
// collapse of tile it released, so three slots would do; four leave a margin.
constexpr int kNQ = 4;
constexpr int kNY = 8;   // slots of the norm's exchange of sums of y^2
static_assert(kNY * kCS * kTMT <= kTMT * kMaxFusedHs, "the norm's sums fit in the f buffer");
constexpr int kBarXFull = 0, kBarRecv = 3, kBarPre = kBarRecv + kNQ, kBarSink = kBarPre + kNQ,
              kBarWFull = kBarSink + 1, kBarSinkDone = kBarWFull + 1, kBarFFull = kBarSinkDone + 1,
              kBarXReady = kBarFFull + 1, kBarYss = kBarXReady + 3, kNumBars = kBarYss + kNY;
// kBarXReady: per stage; kBarYss: per exchange slot, the branch-input norm's sums of y^2
enum WaitSite : unsigned {
    kSiteWFull = 1, kSiteXFull, kSiteRecv, kSitePre, kSiteSink, kSiteDrain, kSiteSinkDone, kSiteYss
};

// Compute-warp map.  Warp w runs on SM sub-partition w%4, whose TMEM lane quarter it
// reads.  Persistent variant: sub-partition q takes row group q&1 and column half q>>1,
// and warpgroup w/4 half of the tile's token slots, so each x value of a stage is
// read by two warps.  Decode variant (fn_w in shared memory, mostly one-token tiles):
// four row groups (w%4) by two column halves (w/4), every warp on all token slots.
template <bool PERSIST>
struct WM {
    static constexpr int RG = PERSIST ? 2 : 4;   // row groups
    static constexpr int TW = PERSIST ? 2 : 1;   // warp token groups
};

// HEAD: the gated-head trunk exit, whose rows equal its streams (pre gates only).
template <int S, bool HEAD = false, int RG = 4>
struct CG {
    static constexpr int R = HEAD ? S : (2 + S) * S;
    static constexpr int RP = (R + RG - 1) / RG * RG;      // rows padded to the row groups
    static constexpr int B = RP / RG;                       // rows per compute warp
    static constexpr int RV = (R + 1 + 3) / 4 * 4;          // exchange stride: R dots + sum of squares
    static constexpr int WQ = 4 * B;                        // fn_w floats per thread per column group
};

// NT = token slots per half-warp (a tile holds up to 2*TW*NT tokens, one owner CTA
// each).  The warps of row group g sum the squares of slots g, g+RG, ...: NSS values
// per thread.
template <int S, int NT, bool HEAD = false, int RG = 4>
struct CT {
    static constexpr int B = CG<S, HEAD, RG>::B;
    static constexpr int NSS = (NT + RG - 1) / RG;
    static constexpr int NV = NT * B + NSS;                 // per-thread values before the reduce-scatter
    static constexpr int NVP = (NV + 15) / 16 * 16;
    static constexpr int VPL = NVP / 16;                    // per-lane values after it
};

struct Lay {   // shared-memory layout in bytes
    int stage_bytes, nst, off_w, off_recv, off_pre, off_sink, off_coef, off_f, off_yss, off_bar, off_misc, total;
};

template <int S, bool PERSIST, bool HEAD>
__host__ __device__ inline Lay make_lay(int LK)
{
    using G = CG<S, HEAD, WM<PERSIST>::RG>;
    Lay L;
    L.stage_bytes = kTMT * LK * 4;
    L.nst = PERSIST ? kNstPersist : 1;
    int o = L.nst * L.stage_bytes;
    L.off_w = o;
    if (!PERSIST)
        o += G::RP * LK * 4;
    L.off_recv = o;                  // [kNQ slots][16 source CTAs][2 column halves][RV]
    o += kNQ * 2 * kCS * G::RV * 4;
    L.off_pre = o;                   // [kNQ slots][16 tokens][4]: the tile's pre gates
    o += kNQ * kTMT * 4 * 4;
    L.off_sink = o;                  // [16 tokens][16]: the comb blocks this CTA scales
    o += kTMT * 16 * 4;
    L.off_coef = o;                  // [2][16 tokens][s + s*s]: fused post -> pre, two tiles' post/comb
    o += (2 * kTMT * (S + S * S) * 4 + 127) / 128 * 128;
    L.off_f = o;                     // [16 tokens][hs <= 256]: fused post -> pre, the tile's slice of f
    o += kTMT * kMaxFusedHs * 4;
    // [kNY slots][16 source CTAs][16 tokens]: the norm's sums of y^2, over the f buffer
    // (the norm runs in the pre-chain mode only, which has no f)
    L.off_yss = L.off_f;
    L.off_bar = o;
    o += kNumBars * 8;
    L.off_misc = o;                  // TMEM address, abort flag, TMA loads issued per stage, f loads
    o += 32;
    L.total = o;
    return L;
}

struct Params {
    // Both maps see a [rows][s][d] tensor as 4-D (hc, d/hc, s, rows), hc = hs/hsc a
    // divisor of hs of at most 256 floats, so a box of (hc, hsc, s, n) is one CTA's
    // column slice of n rows and every box dimension stays within TMA's 256 limit.
    CUtensorMap tmap_x;   // x: rows = tokens, box n = tm_tile
    CUtensorMap tmap_w;   // fn_w: rows = R, box n = R
    CUtensorMap tmap_f;   // fused post -> pre: f as [T][1][d], box (hc, hsc, 1, tm_tile)
    CUtensorMap tmap_xnew;   // fused post -> pre: x_new, boxes as for x
    const float *x, *fn_w, *scale, *base;
    float *pre, *post, *comb, *y;
    // Fused post -> pre (x_new != nullptr): x holds the previous site's input state,
    // and each tile is first turned into x' = post_prev . f + comb_prev^T x (written
    // to x_new), on which this site's pre-chain then runs.
    const float *f, *post_prev, *comb_prev;
    float *x_new;
    // Branch-input norm (z != nullptr; pre-chain mode only): z = y * rsqrt(mean(y^2) +
    // eps_norm) * norm_w and, if q != nullptr, its Q8_0 pair (blocks of 32 columns).
    const float *norm_w;
    float *z;
    signed char *q;
    float *q_scale;
    float eps_norm, inv_d;   // inv_d = 1 / d
    StatusBlock *status;
    unsigned long long *stamps;   // phase stamps (HC_STAMPS builds), else null
    int T, d, hs, hsc, LK, NJ, iters, tm_tile, ntiles;
    int y_rows;   // rows of y (the call's T): bounds of the bounds-checked build's y stores
    float eps, invK;   // invK = 1 / (s*d)
};

// Phase stamp of tile `it`, event `ev`, by CTAs 0 and 8 of cluster 0 (HC_STAMPS builds only).
#ifdef HC_STAMPS
__device__ __forceinline__ void stamp_at(const Params &p, int cid, uint32_t rank, int it, int ev)
{
    if (p.stamps && cid == 0 && (rank & 7u) == 0u && it >= 0 && it < kStampTiles)
        p.stamps[((size_t)(rank >> 3) * kStampTiles + it) * kStampEvents + ev] = ptx::globaltimer();
}
#define HC_STAMP(it, ev) stamp_at(p, cid, rank, (it), (ev))
#else
#define HC_STAMP(it, ev) \
    do {                 \
    } while (0)
#endif

// Bounded wait on an mbarrier phase.  honor_abort = false is used only to let
// this CTA's own bulk copies land before it exits.
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      StatusBlock *sb, unsigned site, bool honor_abort = true)
{
    auto probe = [&]() {
        return CLUSTER_SCOPE ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
    };
    if (probe())
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (probe())
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
            if (ptx::globaltimer() - t0 > kWaitLimitNs) {
                report_error(sb, kDevWaitTimeout, site);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Bounded wait done by lane 0 of a warp; every lane gets the same answer.  The
// acquire lane 0 performs, followed by __syncwarp, orders the other lanes'
// later reads after the arrivals it observed.
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool warp_wait(int lane, uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          StatusBlock *sb, unsigned site)
{
    bool ok = true;
    if (lane == 0)
        ok = wait_bar<CLUSTER_SCOPE>(bar, parity, abort_flag, sb, site);
    ok = __shfl_sync(kFull, ok, 0);
    __syncwarp();
    return ok;
}

// One level of the xor reduce-scatter over the 16 K-groups of a half-warp:
// lanes whose `M` bit is clear keep the lower half of the list, the others the
// upper half, and each adds its partner's copy of the half it keeps.
template <int N, int M>
__device__ __forceinline__ void rs_level(float *v, int kg)
{
    constexpr int H = N / 2;
    const bool hi = (kg & M) != 0;
#pragma unroll
    for (int k = 0; k < H; ++k) {
        const float a = v[k], b = v[k + H];
        const float send = hi ? a : b;
        const float keep = hi ? b : a;
        v[k] = keep + __shfl_xor_sync(kFull, send, M);
    }
}
// After it, lane kg holds the half-warp sums of values [VPL*kg, VPL*kg + VPL).
template <int N>
__device__ __forceinline__ void reduce_scatter16(float *v, int kg)
{
    rs_level<N, 8>(v, kg);
    rs_level<N / 2, 4>(v, kg);
    rs_level<N / 4, 2>(v, kg);
    rs_level<N / 8, 1>(v, kg);
}

// Pairwise sum of n register values (a fixed tree: short dependency chain).
template <int N>
__device__ __forceinline__ float tree_sum(const float *v)
{
    if constexpr (N == 1) {
        return v[0];
    } else {
        return tree_sum<N / 2>(v) + tree_sum<N - N / 2>(v + N / 2);
    }
}

// Sinkhorn on an S x S matrix held in registers: `iters` rounds of dividing
// each row by (row sum + eps), then each column by (column sum + eps).  Each
// division is a multiply by the hardware's approximate reciprocal
// (`rcp.approx.ftz.f32`, within 1 ulp; a sum of positive terms plus eps is never
// subnormal), one instruction on the Sinkhorn's serial chain; the Sinkhorn's error
// budget against the float64 oracle is 1e-4.
template <int S>
__device__ __forceinline__ void sinkhorn_regs(float *c, int iters, float eps)
{
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const float inv = ptx::rcp_approx(tree_sum<S>(c + j * S) + eps);
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
            const float inv = ptx::rcp_approx(tree_sum<S>(col) + eps);
#pragma unroll
            for (int j = 0; j < S; ++j)
                c[j * S + k] *= inv;
        }
    }
}

// The sums of squares of the token slots this warp owns (slot i with i % RG == rg),
// from the x registers of slots i0 .. i0+NH-1 that the dots just loaded: lo then hi.
template <int RG, int NSS, int NH>
__device__ __forceinline__ void squares_step(float2 (&ssa)[NSS], const float4 (&xv)[NH], int i0, int rg)
{
#pragma unroll
    for (int i = 0; i < NH; ++i) {
        if ((i0 + i) % RG == rg) {
            const int m = (i0 + i) / RG;
            const float2 lo = make_float2(xv[i].x, xv[i].y), hi = make_float2(xv[i].z, xv[i].w);
            ssa[m] = ptx::ffma2(lo, lo, ssa[m]);
            ssa[m] = ptx::ffma2(hi, hi, ssa[m]);
        }
    }
}

// One 64-column group of the dots, fn_w from shared memory (decode variant): lane kg's
// two column pairs (2kg, 2kg+1 and 32+2kg, 33+2kg: each half-warp load is 128
// contiguous bytes) of the NT token slots of this half-warp, times this warp's B rows,
// as packed float32 FMAs (acc = (even-column sum, odd-column sum)); plus this warp's
// sums of squares.
template <int B, int NT, int RG, int NSS>
__device__ __forceinline__ void dots_step_smem(float2 (&acc)[NT][B], float2 (&ssa)[NSS],
                                               const float (&w)[4 * B], uint32_t xs_addr, uint32_t cofs,
                                               int lk4, int rg)
{
    constexpr int NH = NT > 4 ? 4 : NT;   // token slots per half (fewer live x registers)
#pragma unroll
    for (int i0 = 0; i0 < NT; i0 += NH) {
        float4 xv[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) {
            const float2 a = ptx::lds64(xs_addr + (uint32_t)((i0 + i) * lk4) + cofs);
            const float2 b = ptx::lds64(xs_addr + (uint32_t)((i0 + i) * lk4) + cofs + 128u);
            xv[i] = make_float4(a.x, a.y, b.x, b.y);
        }
        // The first column pair of every slot and row, then the second: consecutive
        // packed FMAs never depend on each other.
#pragma unroll
        for (int i = 0; i < NH; ++i)
#pragma unroll
            for (int r = 0; r < B; ++r)
                acc[i0 + i][r] = ptx::ffma2(make_float2(xv[i].x, xv[i].y), make_float2(w[4 * r], w[4 * r + 1]),
                                            acc[i0 + i][r]);
#pragma unroll
        for (int i = 0; i < NH; ++i)
#pragma unroll
            for (int r = 0; r < B; ++r)
                acc[i0 + i][r] = ptx::ffma2(make_float2(xv[i].z, xv[i].w), make_float2(w[4 * r + 2], w[4 * r + 3]),
                                            acc[i0 + i][r]);
        squares_step<RG, NSS, NH>(ssa, xv, i0, rg);
    }
}

// The same column group with fn_w from TMEM (persistent variant).  The thread's
// 4*B values of the group sit at columns taddr .. taddr+4B: its first column pair for
// each of its B rows, then its second; each pair block is one TMEM load of 2*B
// registers.  Same FMA order per accumulator as dots_step_smem.
template <int B, int NT, int RG, int NSS>
__device__ __forceinline__ void dots_step_tmem(float2 (&acc)[NT][B], float2 (&ssa)[NSS], uint32_t taddr,
                                               uint32_t xs_addr, uint32_t cofs, int lk4, int rg)
{
    float2 xp[NT];
    float w[2 * B];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
#pragma unroll
        for (int i = 0; i < NT; ++i)
            xp[i] = ptx::lds64(xs_addr + (uint32_t)(i * lk4) + cofs + 128u * (uint32_t)p);
        ptx::tmem_ld_issue<2 * B>(taddr + (uint32_t)(2 * B * p), w);
        ptx::tmem_ld_wait_regs<2 * B>(w);
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int r = 0; r < B; ++r)
                acc[i][r] = ptx::ffma2(xp[i], make_float2(w[2 * r], w[2 * r + 1]), acc[i][r]);
#pragma unroll
        for (int i = 0; i < NT; ++i)
            if (i % RG == rg)
                ssa[i / RG] = ptx::ffma2(xp[i], xp[i], ssa[i / RG]);
    }
}

template <int S, bool PERSIST, int NT, bool HEAD>
__global__ void __launch_bounds__(kThreads, 1) hc_pre_cluster_kernel(const __grid_constant__ Params p)
{
    constexpr int RG = WM<PERSIST>::RG;
    using G = CG<S, HEAD, RG>;
    using C = CT<S, NT, HEAD, RG>;
    static_assert(2 * WM<PERSIST>::TW * NT <= kTMT, "token slots");
    extern __shared__ __align__(128) unsigned char smem[];
    const Lay L = make_lay<S, PERSIST, HEAD>(p.LK);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = (int)ptx::cluster_id_x(), ncl = (int)ptx::ncluster_x();
    float *stages = reinterpret_cast<float *>(smem);
    float *wsm = reinterpret_cast<float *>(smem + L.off_w);
    float *recv = reinterpret_cast<float *>(smem + L.off_recv);
    float *preb = reinterpret_cast<float *>(smem + L.off_pre);
    float *sinkbuf = reinterpret_cast<float *>(smem + L.off_sink);
    float *coefs = reinterpret_cast<float *>(smem + L.off_coef);
    float *fbuf = reinterpret_cast<float *>(smem + L.off_f);
    volatile int *f_issued = reinterpret_cast<volatile int *>(smem + L.off_misc + 20);
    const uint32_t bar0 = ptx::smem_u32(smem + L.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L.off_misc + 8);   // per stage
    StatusBlock *sb = p.status;
    const int stage_floats = L.stage_bytes / 4;
    const int njh = (p.NJ + 1) / 2;   // column groups of the first half (the second gets the rest)
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto tile_tokens = [&](int it, int &t0, int &tm) {
        t0 = (cid + it * ncl) * p.tm_tile;
        tm = min(p.tm_tile, p.T - t0);
    };
    auto tile_exists = [&](int it) { return cid + it * ncl < p.ntiles; };
    const uint32_t hs_bytes = (uint32_t)p.hs * 4u;
    // TMA-load tile `it` into its stage (one instruction; the stage must be free).
    // A partial last tile still moves a whole box: rows past T arrive as zeros.
    const uint32_t tile_box_bytes = (uint32_t)(p.tm_tile * S) * hs_bytes;
    auto load_tile = [&](int it) {   // lane 0 of one warp
        const int s = it % L.nst;
        int t0, tm;
        tile_tokens(it, t0, tm);
        ptx::mbar_arrive_expect_tx(BAR(kBarXFull + s), tile_box_bytes);
        ptx::tma_load_4d(ptx::smem_u32(stages + s * stage_floats), &p.tmap_x, 0, (int)rank * p.hsc, 0,
                         t0, BAR(kBarXFull + s));
        issued[s] = issued[s] + 1;
    };
    // Fused post -> pre: TMA-load tile it's slice of f into the f buffer (one thread).
    auto load_f = [&](int it) {
        int t0, tm;
        tile_tokens(it, t0, tm);
        ptx::mbar_arrive_expect_tx(BAR(kBarFFull), (uint32_t)p.tm_tile * hs_bytes);
        ptx::tma_load_4d(ptx::smem_u32(fbuf), &p.tmap_f, 0, (int)rank * p.hsc, 0, t0, BAR(kBarFFull));
        *f_issued = *f_issued + 1;
    };
    // Branch-input norm (p.z set), by 128 threads ct = 0..127: thread (t = ct / 8,
    // hb = ct % 8) owns float4 columns hb, hb + 8, ... of token t's slice of y (in the
    // persistent variant exactly the columns its collapse wrote).  (1) ss: its sum of y^2
    // over them in column order (the persistent collapse accumulates it as it writes y;
    // the decode variant reads y back); (2) norm_send: an xor tree over the token's eight
    // threads, then that CTA sum to every CTA of the cluster (st.async, counted on slot
    // it % kNY of kBarYss); (3) norm_finish, once all 16 CTAs' sums are in: r = rsqrt(their
    // sum, CTA c into accumulator c % 4 in CTA order, then (a0 + a1) + (a2 + a3), / d +
    // eps_norm), then z = y * r * norm_w over the thread's columns and, with q, the Q8_0
    // pair of each block of 32 (one block = the m-th float4 of the token's eight threads;
    // d / 16 % 32 == 0 keeps blocks inside a CTA's slice).  The persistent collapse
    // finishes tile it after sending tile it + 1.  Slot reuse: a CTA can send tile
    // it + kNY's sums only after collapsing it, which needs this CTA's partials of that
    // tile, so this CTA's stage refill after collapsing tile it + kNY - 3 -- later than
    // its finish of tile it.
    float *yss = reinterpret_cast<float *>(smem + L.off_yss);
    auto norm_send = [&](int it, int ct, float ss) {
        const int q = it % kNY;
        ss += __shfl_xor_sync(kFull, ss, 1);
        ss += __shfl_xor_sync(kFull, ss, 2);
        ss += __shfl_xor_sync(kFull, ss, 4);
        if (ct == 0)
            ptx::mbar_arrive_expect_tx(BAR(kBarYss + q), (uint32_t)(kCS * kTMT * 4));
        if ((ct & 7) == 0) {
            const uint32_t dst = ptx::smem_u32(yss + (q * kCS + (int)rank) * kTMT + (ct >> 3));
            for (int c = 0; c < kCS; ++c)
                ptx::st_async_f32(ptx::mapa(dst, (uint32_t)c), ss, ptx::mapa(BAR(kBarYss + q), (uint32_t)c));
        }
    };
    auto norm_finish = [&](int it, int ct, uint32_t nb) -> bool {
        const int q = it % kNY;
        int t0, tm;
        tile_tokens(it, t0, tm);
        const int t = ct >> 3, hb = ct & 7;
        const bool act = t < tm;
        const int h4n = p.hs / 4;
        const size_t col0 = (size_t)rank * p.hs;
        const size_t row = (size_t)(t0 + (act ? t : 0)) * p.d + col0;
        bool got = true;
        if (ct == 0) {
            got = wait_bar<true>(BAR(kBarYss + q), (it / kNY) & 1, abort_flag, sb, kSiteYss);
            if (!got)   // giving up: still let the sums already on their way land before exit
                wait_bar<true>(BAR(kBarYss + q), (it / kNY) & 1, abort_flag, sb, kSiteDrain, false);
        }
        if (!ptx::named_bar_and(nb, 128, got))
            return false;
        float a4[4] = {0.f, 0.f, 0.f, 0.f};   // CTA c into a4[c % 4], in CTA order
#pragma unroll
        for (int c = 0; c < kCS; ++c)
            a4[c & 3] += yss[(q * kCS + c) * kTMT + t];
        const float r = rsqrtf(((a4[0] + a4[1]) + (a4[2] + a4[3])) * p.inv_d + p.eps_norm);
#pragma unroll 8   // every load of the pass in flight together (one round trip to L2)
        for (int m = 0; m < h4n / 8; ++m) {
            const int h4 = hb + 8 * m;
            float4 zv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (act) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.y + row + 4 * h4));
                const float4 w = __ldg(reinterpret_cast<const float4 *>(p.norm_w + col0 + 4 * h4));
                zv = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
                *reinterpret_cast<float4 *>(p.z + row + 4 * h4) = zv;
            }
            if (p.q) {
                float amax = fmaxf(fmaxf(fabsf(zv.x), fabsf(zv.y)), fmaxf(fabsf(zv.z), fabsf(zv.w)));
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));
                if (act) {
                    const float sc = __fdiv_rn(amax, 127.0f);
                    const float inv = sc != 0.0f ? __frcp_rn(sc) : 0.0f;
                    auto code = [&](float a) {
                        return (signed char)fminf(fmaxf(roundf(__fmul_rn(a, inv)), -127.0f), 127.0f);
                    };
                    *reinterpret_cast<char4 *>(p.q + row + 4 * h4) =
                        make_char4(code(zv.x), code(zv.y), code(zv.z), code(zv.w));
                    if (hb == 0)
                        p.q_scale[(row + 32 * m) / 32] = sc;
                }
            }
        }
        return true;
    };
    // The decode variant's whole norm of its one tile (y written by all compute warps
    // and made visible by a barrier before this call).
    auto norm_tile = [&](int it, int ct, uint32_t nb) -> bool {
        int t0, tm;
        tile_tokens(it, t0, tm);
        const int t = ct >> 3, hb = ct & 7;
        float ss = 0.f;
        if (t < tm) {
            const float *yrow = p.y + (size_t)(t0 + t) * p.d + (size_t)rank * p.hs;
            for (int h4 = hb; h4 < p.hs / 4; h4 += 8) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(yrow + 4 * h4));
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
        }
        norm_send(it, ct, ss);
        return norm_finish(it, ct, nb);
    };

    // ------------------------------------------------------------------ set-up
    if (threadIdx.x == 0)
        HC_STAMP(0, kEvKernelStart);
    if (PERSIST && threadIdx.x == 0)   // the helper kernel queued behind this one may start now
        ptx::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < L.nst; ++s) {
            ptx::mbar_init(BAR(kBarXFull + s), 1);
            issued[s] = 0;
        }
        *f_issued = 0;
        for (int q = 0; q < kNQ; ++q) {
            ptx::mbar_init(BAR(kBarRecv + q), 1);   // armed by this CTA; data by remote stores
            ptx::mbar_init(BAR(kBarPre + q), 1);
        }
        ptx::mbar_init(BAR(kBarSink), 1);
        ptx::mbar_init(BAR(kBarWFull), 1);
        ptx::mbar_init(BAR(kBarSinkDone), 1);
        ptx::mbar_init(BAR(kBarFFull), 1);
        for (int s = 0; s < kNstPersist; ++s)
            ptx::mbar_init(BAR(kBarXReady + s), 1);   // fused persistent: the stage holds x'
        for (int q = 0; q < kNY; ++q)
            ptx::mbar_init(BAR(kBarYss + q), 1);      // armed by this CTA; sums by remote stores
        // A non-zero status word (an earlier launch on this workspace timed out) makes
        // this launch skip its work: 2 marks the skip.  The word only changes 2 s into a
        // launch, so every CTA of the grid reads the same.
        *abort_flag = *reinterpret_cast<volatile unsigned *>(&sb->code) != 0u ? 2 : 0;
        ptx::fence_mbar_init_cluster();
    }
    if (!PERSIST && warp < kNCW) {   // padding rows of the staged fn_w slice are zero
        for (int e = threadIdx.x; e < (G::RP - G::R) * p.LK; e += kComputeThreads)
            wsm[G::R * p.LK + e] = 0.f;
    }
    if (PERSIST && warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    __syncwarp();
    if (PERSIST)
        ptx::tmem_fence_before_sync();
    ptx::cluster_sync_all();   // barriers initialised in every CTA before any remote bulk copy
    if (PERSIST)
        ptx::tmem_fence_after_sync();
    const uint32_t tmem_base = PERSIST ? *tmem_slot : 0u;
    const bool skip = *abort_flag == 2;

    if (skip) {
        // nothing is loaded, computed or written
    } else if (warp < kNCW) {
        ptx::setmaxnreg_inc<kRegsCompute>();
        // -------------------------------------------------------------- compute warps
        // One thread polls each barrier; a named barrier with an AND reduction then
        // hands its answer (and, by the barrier's ordering, what it acquired) to all
        // eight warps, so they always meet the same barriers.
        const int tg = lane >> 4, kg = lane & 15;
        const int sp = warp & 3, wg = warp >> 2;   // sub-partition, warpgroup
        const int rg = PERSIST ? (sp & 1) : sp, half = PERSIST ? (sp >> 1) : wg;
        const int tw = PERSIST ? wg : 0;           // warp token group
        const int j0 = half * njh, nj = half ? p.NJ - njh : njh;
        // TMEM: warp w reads lanes 32*(w%4).. of its sub-partition; both warps of a
        // sub-partition (the two token groups) read the same fn_w values there.
        const uint32_t trow = tmem_base + ((uint32_t)(32 * sp) << 16);
        if (threadIdx.x == 0) {
            // fn_w slice (the persistent variant stages it in stages 1-2, so tile 0
            // can land in stage 0 meanwhile), then the first tile.
            ptx::prefetch_tmap(&p.tmap_x);
            ptx::prefetch_tmap(&p.tmap_w);
            float *wdst = PERSIST ? stages + stage_floats : wsm;
            ptx::mbar_arrive_expect_tx(BAR(kBarWFull), (uint32_t)(G::R * S) * hs_bytes);
            ptx::tma_load_4d(ptx::smem_u32(wdst), &p.tmap_w, 0, (int)rank * p.hsc, 0, 0,
                             BAR(kBarWFull));
            load_tile(0);   // every cluster has at least one tile
            if (p.x_new && !PERSIST)   // the persistent variant's collapse warps load f
                load_f(0);
        }
        bool ok = ptx::named_bar_and(
            1, kComputeThreads, threadIdx.x != 0 || wait_bar<false>(BAR(kBarWFull), 0, abort_flag, sb, kSiteWFull));
        if (PERSIST && ok) {
            // This thread's fixed fn_w values -> its TMEM lane (written by token group 0,
            // read by both): column group jj at columns jj*WQ .., row r's first column
            // pair (2kg, 2kg+1 of the group) at 2r, 2r+1 and its second (32+2kg, 33+2kg)
            // at 2B+2r, 2B+2r+1 (the layout dots_step_tmem reads).
            const float *wstage = stages + stage_floats;
            if (tw == 0) {
                for (int jj = 0; jj < nj; ++jj) {
                    const int c = 64 * (j0 + jj) + 2 * kg;
                    float a[G::WQ];
#pragma unroll
                    for (int r = 0; r < G::B; ++r) {
                        const int row = rg * G::B + r;
                        float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
                        if (row < G::R) {
                            v0 = *reinterpret_cast<const float2 *>(wstage + row * p.LK + c);
                            v1 = *reinterpret_cast<const float2 *>(wstage + row * p.LK + c + 32);
                        }
                        a[2 * r] = v0.x;
                        a[2 * r + 1] = v0.y;
                        a[2 * G::B + 2 * r] = v1.x;
                        a[2 * G::B + 2 * r + 1] = v1.y;
                    }
#pragma unroll
                    for (int m = 0; m < G::B; ++m)
                        ptx::tmem_st4(trow + (uint32_t)(jj * G::WQ + 4 * m), a + 4 * m);
                }
                ptx::tmem_wait_st();
            }
            ptx::tmem_fence_before_sync();
            ptx::named_bar_sync(1, kComputeThreads);
            ptx::tmem_fence_after_sync();
            // Stages 1 and 2 are free now.
            if (threadIdx.x == 0)
                for (int it = 1; it < L.nst && tile_exists(it); ++it)
                    load_tile(it);
        }

        // Decode variant: collapse its one tile once the owners' pre gates are in.
        auto collapse = [&](int itc) -> bool {
            const int q = itc % kNQ;
            const bool got =
                threadIdx.x != 0 || wait_bar<true>(BAR(kBarPre + q), (itc / kNQ) & 1, abort_flag, sb, kSitePre);
            if (!ptx::named_bar_and(1, kComputeThreads, got))
                return false;
            if (threadIdx.x == 0)
                HC_STAMP(itc, kEvPreArrived);
            int t0, tm;
            tile_tokens(itc, t0, tm);
            const int s = itc % L.nst;
            const uint32_t xs_base = ptx::smem_u32(stages + s * stage_floats);
            const uint32_t pre_base = ptx::smem_u32(preb + q * kTMT * 4);
            const int h4n = p.hs / 4;
            for (int e = threadIdx.x; e < kTMT * h4n; e += kComputeThreads) {
                const int t = e / h4n, h4 = e - t * h4n;
                if (t >= tm)
                    break;
                const float4 pv = ptx::lds128(pre_base + 16u * (uint32_t)t);
                const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
                const uint32_t xa = xs_base + 4u * (uint32_t)(t * p.LK + 4 * h4);
                float4 xv = ptx::lds128(xa);
                float4 a = make_float4(pr[0] * xv.x, pr[0] * xv.y, pr[0] * xv.z, pr[0] * xv.w);
#pragma unroll
                for (int k = 1; k < S; ++k) {
                    xv = ptx::lds128(xa + 4u * (uint32_t)(k * p.hs));
                    a.x = fmaf(pr[k], xv.x, a.x);
                    a.y = fmaf(pr[k], xv.y, a.y);
                    a.z = fmaf(pr[k], xv.z, a.z);
                    a.w = fmaf(pr[k], xv.w, a.w);
                }
                store_checked(reinterpret_cast<float4 *>(p.y), ((size_t)(t0 + t) * p.d + (size_t)rank * p.hs + 4 * h4) / 4,
                              (size_t)p.y_rows * p.d / 4, a, p.status, kStoreY);
            }
            if (threadIdx.x == 0)
                HC_STAMP(itc, kEvCollapsed);
            return true;
        };

        // Persistent variant: the two warpgroups (token groups) wait for tiles on
        // their own barriers, and warpgroup 1 starts once warpgroup 0 has done its
        // first dots, so one reduces and ships while the other runs its FMAs.  In its
        // fused post -> pre mode the collapse warps transform each tile (x -> x') and
        // the compute warps wait for that instead of the load.  The decode variant
        // keeps all eight warps together: its collapse, and in fused mode its tile
        // transform, need them all.
        const bool fused = p.x_new != nullptr;
        const bool tf_here = fused && !PERSIST;   // these warps transform the tile
        const bool split = PERSIST;
        const uint32_t tbar = split ? kNbGroup0 + (uint32_t)wg : kNbCompute;
        const uint32_t tthreads = split ? kComputeThreads / 2 : kComputeThreads;
        const int tpoll = split ? wg * (kComputeThreads / 2) : 0;   // the thread that polls
        bool arrived = !(split && wg == 0);
        if (split && wg == 1)
            ptx::named_bar_sync(kNbStagger, kComputeThreads);
        const int lk4 = p.LK * 4;
        // Fused post -> pre: this thread's share of the next tile's post/comb (at most
        // 16 tokens x (s + s*s) values over the 256 compute threads).
        constexpr int NC = S + S * S;
        constexpr int kCoefPerThread = (kTMT * NC + kComputeThreads - 1) / kComputeThreads;
        float cpre[kCoefPerThread];
        auto load_coefs = [&](int itn, float (&c)[kCoefPerThread]) {
            int t0n, tmn;
            tile_tokens(itn, t0n, tmn);
#pragma unroll
            for (int m = 0; m < kCoefPerThread; ++m) {
                const int e = threadIdx.x + m * kComputeThreads;
                c[m] = 0.f;
                if (e < tmn * NC) {
                    const int t = e / NC, cc = e - (e / NC) * NC;
                    c[m] = cc < S ? __ldg(p.post_prev + (size_t)(t0n + t) * S + cc)
                                  : __ldg(p.comb_prev + (size_t)(t0n + t) * S * S + (cc - S));
                }
            }
        };
        int it = 0;
        for (; ok; ++it) {
            if (!tile_exists(it))
                break;
            const int s = it % L.nst, u = it / L.nst;
            const int xbar = (PERSIST && fused) ? kBarXReady + s : kBarXFull + s;
            ok = ptx::named_bar_and(
                tbar, tthreads,
                (int)threadIdx.x != tpoll ||
                    (wait_bar<false>(BAR(xbar), u & 1, abort_flag, sb, kSiteXFull) &&
                     (!tf_here || wait_bar<false>(BAR(kBarFFull), it & 1, abort_flag, sb, kSiteXFull))));
            if (!ok)
                break;
            if (threadIdx.x == 0)   // compute stamps: warpgroup 0
                HC_STAMP(it, kEvStageReady);
            int t0, tm;
            tile_tokens(it, t0, tm);
            if (tf_here) {
                // The previous site's hc_post on this tile, in place: thread e owns the
                // 4 columns h4 of token t in every stream, reads x_prev, writes x' (the
                // same operations, in the same order, as hc_post_kernel).  The tile's
                // post/comb came into registers during the previous tile (cpre), its f
                // slice by TMA.
                if (it == 0)
                    load_coefs(it, cpre);
#pragma unroll
                for (int m = 0; m < kCoefPerThread; ++m) {
                    const int e = threadIdx.x + m * kComputeThreads;
                    if (e < tm * NC)
                        coefs[e] = cpre[m];
                }
                ptx::named_bar_sync(kNbCompute, kComputeThreads);
                // Thread -> (token t = tid / 16, columns h4 = tid % 16 + 16 m): one token's
                // coefficients per thread, loaded once.
                float *xs = stages + s * stage_floats;
                const int h4n = p.hs / 4;
                const int t = threadIdx.x >> 4;
                if (t < tm) {
                    float cf[NC];
#pragma unroll
                    for (int c = 0; c < NC; ++c)
                        cf[c] = coefs[t * NC + c];
                    for (int h4 = threadIdx.x & 15; h4 < h4n; h4 += 16) {
                        float4 *xt = reinterpret_cast<float4 *>(xs + t * p.LK + 4 * h4);
                        const float4 fv = *reinterpret_cast<const float4 *>(fbuf + t * p.hs + 4 * h4);
                        float4 xv[S];
#pragma unroll
                        for (int j = 0; j < S; ++j)
                            xv[j] = xt[j * h4n];
#pragma unroll
                        for (int k = 0; k < S; ++k) {
                            const float pk = cf[k];
                            float4 o = make_float4(pk * fv.x, pk * fv.y, pk * fv.z, pk * fv.w);
#pragma unroll
                            for (int j = 0; j < S; ++j) {
                                const float cc = cf[S + j * S + k];
                                o.x = fmaf(cc, xv[j].x, o.x);
                                o.y = fmaf(cc, xv[j].y, o.y);
                                o.z = fmaf(cc, xv[j].z, o.z);
                                o.w = fmaf(cc, xv[j].w, o.w);
                            }
                            xt[k * h4n] = o;
                        }
                    }
                }
                ptx::fence_proxy_async_smem();   // TMA reads the stage (store) and refills it later
                ptx::named_bar_sync(kNbCompute, kComputeThreads);
                if (threadIdx.x == 0) {   // x' of this tile -> the new state, one TMA store
                    ptx::tma_store_4d(&p.tmap_xnew, 0, (int)rank * p.hsc, 0, t0, ptx::smem_u32(xs));
                    ptx::bulk_commit();
                }
                if (tile_exists(it + 1)) {
                    if (threadIdx.x == 0)
                        load_f(it + 1);
                    load_coefs(it + 1, cpre);
                }
            }
            const int slot0 = (2 * tw + tg) * NT;   // this half-warp's first token slot
            const int ntok = min(NT, max(0, tm - slot0));
            // Byte address of token slot 0 of this half-warp, at this lane's first column group.
            const uint32_t xs_addr = ptx::smem_u32(stages + s * stage_floats + slot0 * p.LK) + 8u * kg;
            const uint32_t ws_addr = ptx::smem_u32(wsm + (rg * G::B) * p.LK) + 8u * kg;

            // Every slot is computed (rows of a stage past the tile's last token hold stale
            // but harmless data, never sent), so the loop has no data-dependent branch.
            float2 acc[NT][G::B];
            float2 ssa[C::NSS];
#pragma unroll
            for (int i = 0; i < NT; ++i)
#pragma unroll
                for (int r = 0; r < G::B; ++r)
                    acc[i][r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int m = 0; m < C::NSS; ++m)
                ssa[m] = make_float2(0.f, 0.f);

            if (PERSIST) {
                // fn_w from TMEM, one column group at a time; the other compute warp
                // of this sub-partition runs its FMAs while this one waits for a load.
                for (int jj = 0; jj < nj; ++jj)
                    dots_step_tmem<G::B, NT, RG, C::NSS>(acc, ssa, trow + (uint32_t)(jj * G::WQ), xs_addr,
                                                         256u * (uint32_t)(j0 + jj), lk4, rg);
            } else {
                for (int jj = 0; jj < nj; ++jj) {
                    const uint32_t cofs = 256u * (uint32_t)(j0 + jj);
                    float w[G::WQ];
#pragma unroll
                    for (int r = 0; r < G::B; ++r) {
                        const float2 v0 = ptx::lds64(ws_addr + (uint32_t)(r * lk4) + cofs);
                        const float2 v1 = ptx::lds64(ws_addr + (uint32_t)(r * lk4) + cofs + 128u);
                        w[4 * r] = v0.x;
                        w[4 * r + 1] = v0.y;
                        w[4 * r + 2] = v1.x;
                        w[4 * r + 3] = v1.y;
                    }
                    dots_step_smem<G::B, NT, RG, C::NSS>(acc, ssa, w, xs_addr, cofs, lk4, rg);
                }
            }
            if (threadIdx.x == 0)
                HC_STAMP(it, kEvDotsDone);
            if (!arrived) {
                ptx::named_bar_arrive(kNbStagger, kComputeThreads);
                arrived = true;
            }

            // Half-warp sums over the 16 K-groups.
            float v[C::NVP];
#pragma unroll
            for (int i = 0; i < NT; ++i)
#pragma unroll
                for (int r = 0; r < G::B; ++r)
                    v[i * G::B + r] = acc[i][r].x + acc[i][r].y;
#pragma unroll
            for (int m = 0; m < C::NSS; ++m)
                v[NT * G::B + m] = ssa[m].x + ssa[m].y;
#pragma unroll
            for (int q = C::NV; q < C::NVP; ++q)
                v[q] = 0.f;
            reduce_scatter16<C::NVP>(v, kg);
            // Each value goes straight to its token's owner CTA (token t of the tile belongs
            // to CTA t), into recv[tile parity][this CTA][column half][row], by an
            // asynchronous remote store that completes on the owner's recv barrier.  (The
            // owner consumed that slot's previous tile before this CTA could ship this one.)
            const int qb = it % kNQ;
            const uint32_t recv_slot = ptx::smem_u32(recv + ((qb * kCS + (int)rank) * 2 + half) * G::RV);
#pragma unroll
            for (int q = 0; q < C::VPL; ++q) {
                const int o = C::VPL * kg + q;
                int i = NT, vid = -1;
                if (o < NT * G::B) {
                    i = o / G::B;
                    const int row = rg * G::B + (o - i * G::B);
                    vid = row < G::R ? row : -1;
                } else if (o < C::NV) {
                    i = rg + RG * (o - NT * G::B);
                    vid = G::R;
                }
                if (vid >= 0 && i < ntok) {
                    const uint32_t t = (uint32_t)(slot0 + i);
                    ptx::st_async_f32(ptx::mapa(recv_slot + 4u * (uint32_t)vid, t), v[q],
                                      ptx::mapa(BAR(kBarRecv + qb), t));
                }
            }
            if (threadIdx.x == 0)
                HC_STAMP(it, kEvShipped);
            if (!PERSIST) {
                if (threadIdx.x == 0)   // the owners will answer with tm pre gates
                    ptx::mbar_arrive_expect_tx(BAR(kBarPre + qb), (uint32_t)(tm * 16));
                if (!(ok = collapse(it)))
                    break;
                if (p.z) {   // the branch-input norm, by warps 0-3 once every y column is written
                    ptx::named_bar_sync(kNbCompute, kComputeThreads);
                    if (warp < 4 && !(ok = norm_tile(it, threadIdx.x, kNbGroup0)))
                        break;
                }
            }
        }
        if (!arrived)
            ptx::named_bar_arrive(kNbStagger, kComputeThreads);
        if (tf_here && threadIdx.x == 0)
            ptx::bulk_wait_all();   // every x' store complete before the CTA can exit
    } else {
        if (warp >= kCollapseWarp0)
            ptx::setmaxnreg_dec<kRegsCollapse>();
        else
            ptx::setmaxnreg_dec<kRegsFinish>();
        if (warp < kSinkWarp) {
            // -------------------------------------------------------------- finisher warps
            // Tile it's token t is owned by CTA t: its finisher (warp 8 + it % 2) sums the
            // 2 x 16 partials, forms the gates, sends pre to every CTA and post to memory,
            // and hands exp(comb logits) to the tile's Sinkhorn CTA (it % 16), whose
            // Sinkhorn warp scales all of the tile's tokens at once, one token per lane.
            // Only a cluster's last tile can be partial, so no later tile's bytes can
            // reach a CTA that owns nothing in this one.
            //
            // A CTA's Sinkhorn buffer is reused 16 tiles later.  Before this finisher sends
            // the gates of tile it, it waits until its CTA's Sinkhorn warp is done with tile
            // it - 8 if that tile was this CTA's: tile it - 8 + 16's exp values can only
            // come once this CTA has shipped it, after collapsing tile it + 4, which needs
            // gates this finisher sends after those of tile it.
            const int f = warp - kFinisherWarp;
            const int grp = lane < S ? 0 : (lane < 2 * S ? 1 : 2);
            const float my_scale = lane < G::R ? p.scale[grp] : 0.f;
            const float my_base = lane < G::R ? p.base[lane] : 0.f;
            for (int it = f; tile_exists(it); it += 2) {
                const int qb = it % kNQ;
                int t0, tm;
                tile_tokens(it, t0, tm);
                const bool own = (int)rank < tm;
                const uint32_t sc = (uint32_t)(it % kCS);
                const int itl = it - kSinkLag;
                if (!HEAD && itl >= 0 && itl % kCS == (int)rank &&
                    !warp_wait<false>(lane, BAR(kBarSinkDone), (itl / kCS) & 1, abort_flag, sb, kSiteSinkDone))
                    break;
                if (lane == 0)
                    ptx::mbar_arrive_expect_tx(BAR(kBarRecv + qb), own ? (uint32_t)(2 * kCS * (G::R + 1) * 4) : 0u);
                if (!warp_wait<true>(lane, BAR(kBarRecv + qb), (it / kNQ) & 1, abort_flag, sb, kSiteRecv)) {
                    // Giving up: still let any partials already on their way land before exit.
                    if (lane == 0)
                        wait_bar<true>(BAR(kBarRecv + qb), (it / kNQ) & 1, abort_flag, sb, kSiteDrain, false);
                    __syncwarp();
                    break;
                }
                if (lane == 0)
                    HC_STAMP(it, kEvPartials);
                if (own) {
                    float val = 0.f;
                    if (lane <= G::R) {
                        float src[2 * kCS];
                        const uint32_t a0 = ptx::smem_u32(recv + qb * 2 * kCS * G::RV + lane);
    #pragma unroll
                        for (int c = 0; c < 2 * kCS; ++c)
                            src[c] = ptx::lds32(a0 + 4u * (uint32_t)(c * G::RV));
                        val = tree_sum<2 * kCS>(src);   // sources and halves in a fixed pairwise order
                    }
                    const float ss = __shfl_sync(kFull, val, G::R);
                    const float rinv = rsqrtf(ss * p.invK + p.eps);
                    const float logit = lane < G::R ? val * rinv * my_scale + my_base : 0.f;
                    // Hardware exp2-based exponential and fast divide (a few ulp each): the
                    // gates sit on the path from the partials to the collapse, and this warp
                    // shares its sub-partition with two FMA-bound compute warps.
                    const float sg = __fdividef(1.f, 1.f + __expf(-logit));
                    const float pre_v = sg + p.eps;
                    // pre gates of this token -> every CTA of the cluster (16 bytes each);
                    // exp(comb logits) -> the Sinkhorn CTA, one value per lane.
                    float4 pv;
                    pv.x = __shfl_sync(kFull, pre_v, 0);
                    pv.y = __shfl_sync(kFull, pre_v, 1 % S);
                    pv.z = __shfl_sync(kFull, pre_v, 2 % S);
                    pv.w = __shfl_sync(kFull, pre_v, 3 % S);
                    if (lane < kCS) {
                        const uint32_t dst = ptx::smem_u32(preb + (qb * kTMT + (int)rank) * 4);
                        ptx::st_async_v4(ptx::mapa(dst, (uint32_t)lane), pv, ptx::mapa(BAR(kBarPre + qb), (uint32_t)lane));
                    }
                    if (!HEAD && lane >= 2 * S && lane < G::R) {
                        const uint32_t dst = ptx::smem_u32(sinkbuf + (int)rank * 16 + (lane - 2 * S));
                        ptx::st_async_f32(ptx::mapa(dst, sc), __expf(logit), ptx::mapa(BAR(kBarSink), sc));
                    }
                    if (lane == 0)
                        HC_STAMP(it, kEvGatesSent);
                    const size_t tok = (size_t)t0 + rank;
                    if (lane < S) {
                        if (p.pre)   // the head's gates are an optional output
                            store_checked(p.pre, tok * S + lane, (size_t)p.T * S, pre_v, p.status, kStorePre);
                    } else if (!HEAD && lane < 2 * S) {
                        store_checked(p.post, tok * S + (lane - S), (size_t)p.T * S, 2.f * sg, p.status, kStorePost);
                    }
                }
                __syncwarp();
            }
        } else if (!HEAD && warp == kSinkWarp) {
            // -------------------------------------------------------------- Sinkhorn warp
            // Tiles rank, rank + 16, ... are this CTA's to normalise: lane t takes token
            // t's S x S block of exp(comb logits) and runs the Sinkhorn in registers.
            for (int it = (int)rank; tile_exists(it); it += kCS) {
                int t0, tm;
                tile_tokens(it, t0, tm);
                if (lane == 0)
                    ptx::mbar_arrive_expect_tx(BAR(kBarSink), (uint32_t)(tm * S * S * 4));
                if (!warp_wait<true>(lane, BAR(kBarSink), (it / kCS) & 1, abort_flag, sb, kSiteSink)) {
                    if (lane == 0)
                        wait_bar<true>(BAR(kBarSink), (it / kCS) & 1, abort_flag, sb, kSiteDrain, false);
                    __syncwarp();
                    break;
                }
                if (lane < tm) {
                    float cm[S * S];
                    const float *src = sinkbuf + lane * 16;
    #pragma unroll
                    for (int q = 0; q < S * S; ++q)
                        cm[q] = src[q];
                    sinkhorn_regs<S>(cm, p.iters, p.eps);
    #pragma unroll
                    for (int q = 0; q < S * S; ++q)
                        store_checked(p.comb, (size_t)(t0 + lane) * S * S + q, (size_t)p.T * S * S, cm[q], p.status,
                                      kStoreComb);
                }
                __syncwarp();
                if (lane == 0) {
                    HC_STAMP(it, kEvSinkDone);
                    ptx::mbar_arrive(BAR(kBarSinkDone));   // the buffer may be refilled
                }
            }
        } else if (PERSIST && warp >= kCollapseWarp0) {
            // -------------------------------------------------------------- collapse warps
            // Tile by tile: wait for the owners' pre gates, write y for this CTA's hidden
            // columns from the tile's stage, then refill the stage with tile it + nst.  The
            // compute warps never wait for gates; only the stage ring links them to these.
            // Fused post -> pre mode: these warps also turn each landed tile into x' in
            // place (the previous site's hc_post), store x' by TMA and release the stage
            // to the compute warps, two tiles ahead of their collapse.
            const int ct = threadIdx.x - kCollapseWarp0 * 32;
            const int h4n = p.hs / 4;
            // Thread -> token t = ct / 8 (its gates or coefficients loaded once) and float4
            // columns h4 = ct % 8 + 8 m: eight threads cover 128 contiguous bytes of a row.
            constexpr int U = 2;   // outputs per thread in flight
            const int t = ct >> 3, hb = ct & 7;
            const bool fused = p.x_new != nullptr;
            constexpr int NC = S + S * S;
            // Fused: tile k's post / comb values (at most 16 tokens x (s + s*s)) into coef
            // buffer k % 2 by asynchronous copies, issued one transform ahead.
            auto load_coefs_c = [&](int k) {
                int t0n, tmn;
                tile_tokens(k, t0n, tmn);
                float *cb = coefs + (k & 1) * (kTMT * NC);
                for (int e = ct; e < tmn * NC; e += kCollapseThreads) {
                    const int tt = e / NC, cc = e - tt * NC;
                    ptx::cp_async4(ptx::smem_u32(cb + e), cc < S ? p.post_prev + (size_t)(t0n + tt) * S + cc
                                                                 : p.comb_prev + (size_t)(t0n + tt) * S * S + (cc - S));
                }
                ptx::cp_async_commit();
            };
            // x -> x' for tile k (the same operations, in the same order, as hc_post_kernel).
            auto transform = [&](int k) -> bool {
                const int s = k % L.nst;
                int t0, tm;
                tile_tokens(k, t0, tm);
                if (ct == 0)
                    HC_STAMP(k, kEvXfStart);
                ptx::cp_async_wait_all();   // this thread's copies of the tile's post / comb
                bool got = true;
                if (ct == 0)
                    got = wait_bar<false>(BAR(kBarXFull + s), (k / L.nst) & 1, abort_flag, sb, kSiteXFull) &&
                          wait_bar<false>(BAR(kBarFFull), k & 1, abort_flag, sb, kSiteXFull);
                if (!ptx::named_bar_and(kNbCollapse, kCollapseThreads, got))
                    return false;
                if (ct == 0)
                    HC_STAMP(k, kEvXfLanded);
                if (t < tm) {   // (the barrier above made every thread's coef copies visible)
                    const float *cb = coefs + (k & 1) * (kTMT * NC);
                    float cf[NC];
    #pragma unroll
                    for (int c = 0; c < NC; ++c)
                        cf[c] = cb[t * NC + c];
                    float *xr = stages + s * stage_floats + t * p.LK;
                    const float *fr = fbuf + t * p.hs;
                    for (int h4 = hb; h4 < h4n; h4 += 8) {
                        float4 *xt = reinterpret_cast<float4 *>(xr + 4 * h4);
                        const float4 fv = *reinterpret_cast<const float4 *>(fr + 4 * h4);
                        float4 xv[S];
    #pragma unroll
                        for (int j = 0; j < S; ++j)
                            xv[j] = xt[j * h4n];
    #pragma unroll
                        for (int kk = 0; kk < S; ++kk) {
                            const float pk = cf[kk];
                            float4 o = make_float4(pk * fv.x, pk * fv.y, pk * fv.z, pk * fv.w);
    #pragma unroll
                            for (int j = 0; j < S; ++j) {
                                const float cc = cf[S + j * S + kk];
                                o.x = fmaf(cc, xv[j].x, o.x);
                                o.y = fmaf(cc, xv[j].y, o.y);
                                o.z = fmaf(cc, xv[j].z, o.z);
                                o.w = fmaf(cc, xv[j].w, o.w);
                            }
                            xt[kk * h4n] = o;
                        }
                    }
                }
                ptx::fence_proxy_async_smem();   // the TMA store reads the stage, a TMA load refills it
                ptx::named_bar_sync(kNbCollapse, kCollapseThreads);
                if (ct == 0) {
                    ptx::tma_store_4d(&p.tmap_xnew, 0, (int)rank * p.hsc, 0, t0, ptx::smem_u32(stages + s * stage_floats));
                    ptx::bulk_commit();
                    ptx::mbar_arrive(BAR(kBarXReady + s));   // the compute warps may read x'
                    HC_STAMP(k, kEvXfDone);
                    if (tile_exists(k + 1))
                        load_f(k + 1);
                }
                if (tile_exists(k + 1))
                    load_coefs_c(k + 1);
                return true;
            };
            int nt = 0;   // the next tile to transform
            bool tok = true;
            if (fused) {
                if (ct == 0)
                    load_f(0);
                load_coefs_c(0);
                for (; tok && nt < 2 && tile_exists(nt); ++nt)
                    tok = transform(nt);
            }
            int ndone = 0;   // tiles collapsed
            for (int it = 0; tok && tile_exists(it); ++it) {
                if (ct == 0 && tile_exists(it + L.nst + 1)) {
                    // The box of the tile whose stage load the next iteration issues, into L2
                    // now, so that load reads L2 (fused: the transform after it waits for it).
                    int t0n, tmn;
                    tile_tokens(it + L.nst + 1, t0n, tmn);
                    ptx::tma_prefetch_l2_4d(&p.tmap_x, 0, (int)rank * p.hsc, 0, t0n);
                }
                if (fused && tile_exists(nt)) {   // nt = it + 2
                    if (!(tok = transform(nt)))
                        break;
                    ++nt;
                }
                const int q = it % kNQ;
                int t0, tm;
                tile_tokens(it, t0, tm);
                bool got = true;
                if (ct == 0) {   // the owners answer with tm pre gates
                    ptx::mbar_arrive_expect_tx(BAR(kBarPre + q), (uint32_t)(tm * 16));
                    got = wait_bar<true>(BAR(kBarPre + q), (it / kNQ) & 1, abort_flag, sb, kSitePre);
                }
                if (!ptx::named_bar_and(kNbCollapse, kCollapseThreads, got))
                    break;
                if (ct == 0)
                    HC_STAMP(it, kEvPreArrived);
                float ssy = 0.f;   // the norm's sum of y^2 over this thread's columns, in column order
                if (t < tm) {
                    const float4 pv = ptx::lds128(ptx::smem_u32(preb + (q * kTMT + t) * 4));
                    const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
                    const uint32_t xrow = ptx::smem_u32(stages + (it % L.nst) * stage_floats + t * p.LK);
                    const size_t y4 = ((size_t)(t0 + t) * p.d + (size_t)rank * p.hs) / 4;   // y row, float4s
                    for (int h0 = hb; h0 < h4n; h0 += 8 * U) {
                        float4 xv[U][S];
    #pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int h4 = min(h0 + 8 * u, h4n - 1);
    #pragma unroll
                            for (int k = 0; k < S; ++k)
                                xv[u][k] = ptx::lds128(xrow + 4u * (uint32_t)(k * p.hs + 4 * h4));
                        }
    #pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int h4 = h0 + 8 * u;
                            if (h4 >= h4n)
                                break;
                            float4 a = make_float4(pr[0] * xv[u][0].x, pr[0] * xv[u][0].y, pr[0] * xv[u][0].z,
                                                   pr[0] * xv[u][0].w);
    #pragma unroll
                            for (int k = 1; k < S; ++k) {
                                a.x = fmaf(pr[k], xv[u][k].x, a.x);
                                a.y = fmaf(pr[k], xv[u][k].y, a.y);
                                a.z = fmaf(pr[k], xv[u][k].z, a.z);
                                a.w = fmaf(pr[k], xv[u][k].w, a.w);
                            }
                            store_checked(reinterpret_cast<float4 *>(p.y), y4 + h4, (size_t)p.y_rows * p.d / 4, a,
                                          p.status, kStoreY);
                            if (p.z) {
                                ssy = fmaf(a.x, a.x, ssy);
                                ssy = fmaf(a.y, a.y, ssy);
                                ssy = fmaf(a.z, a.z, ssy);
                                ssy = fmaf(a.w, a.w, ssy);
                            }
                        }
                    }
                }
                ptx::named_bar_sync(kNbCollapse, kCollapseThreads);
                if (ct == 0)
                    HC_STAMP(it, kEvCollapsed);
                if (ct == 0 && tile_exists(it + L.nst)) {
                    // Fused: tile it's x' store has read the stage (only the stores of
                    // tiles it + 1 and it + 2 may still be pending).
                    if (fused)
                        ptx::bulk_wait_read<2>();
                    load_tile(it + L.nst);
                    HC_STAMP(it, kEvRefilled);
                }
                if (p.z) {   // send this tile's sums, finish the previous tile's norm
                    norm_send(it, ct, ssy);
                    if (it > 0 && !(tok = norm_finish(it - 1, ct, kNbCollapse)))
                        break;
                }
                ++ndone;
            }
            if (p.z && tok && ndone > 0)
                tok = norm_finish(ndone - 1, ct, kNbCollapse);
            if (fused && ct == 0)
                ptx::bulk_wait_all();   // every x' store complete before the CTA can exit
        }
    }

    // ------------------------------------------------------------------ teardown
    __syncwarp();
    if (PERSIST)
        ptx::tmem_fence_before_sync();
    ptx::cluster_sync_all();   // no CTA leaves while another may still write its shared memory
    // Every TMA load this CTA issued (by whichever warp) lands before it exits.
    if (threadIdx.x == 0 && !skip) {
        wait_bar<false>(BAR(kBarWFull), 0, abort_flag, sb, kSiteDrain, false);
        for (int s = 0; s < L.nst; ++s)
            if (issued[s] > 0)
                wait_bar<false>(BAR(kBarXFull + s), (issued[s] - 1) & 1, abort_flag, sb, kSiteDrain, false);
        if (*f_issued > 0)
            wait_bar<false>(BAR(kBarFFull), (*f_issued - 1) & 1, abort_flag, sb, kSiteDrain, false);
    }
    __syncwarp();
    if (PERSIST) {
        ptx::tmem_fence_after_sync();
        if (warp == 0)
            ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------- helper kernel
// The persistent cluster kernel fills only the SMs that 16-CTA clusters can be placed on
// (112 of 152 on a GB300); the others would idle.  The helper kernel runs on them, launched
// right behind the cluster kernel on the same stream with programmatic dependent launch (the
// cluster kernel lets it start at once).  It takes whole 8-token tiles from the end of the
// batch, never the cluster kernel's tokens, and each of its CTAs plays the 16 CTAs of a
// cluster in turn, with the decode variant's arithmetic in the decode variant's order, so
// every token's outputs are the same bits whichever kernel computed them:
//  * phase 1, slice c = 0..15 (hidden columns [c*hs, (c+1)*hs) of every stream): the fn_w
//    slice into TMEM (staged through shared memory while the previous slice is in use, then
//    copied by each thread into its own lane); then for each of the CTA's tiles the tile's
//    slice by TMA (three buffers, two steps ahead; fused mode: with the f slice, then the
//    previous site's hc_post in place and the x' slice stored by TMA), the eight warps' dots,
//    the 16-lane reduce-scatter, and the two column halves' partials of every token into the
//    workspace.  In the pre-chain mode the warps never wait for one another here: the last
//    warp done with a buffer refills it;
//  * phase 2: per token, the 2 x 16 partials in the finisher's order, the gates, pre/post;
//    the Sinkhorn, one token per thread; then y over all d columns from x (fused: x') read
//    back from memory.
// Waits are bounded as in the cluster kernel.  Before it exits the helper waits for the
// cluster kernel to complete (griddepcontrol.wait), so whatever the stream runs next sees
// the outputs of both.
constexpr int kHT = 8;                         // tokens per helper tile
constexpr int kHNT = 4;                        // token slots per half-warp: two half-warps, 8 tokens
constexpr int kHThreads = kComputeThreads;     // the eight compute warps of the decode variant
constexpr int kHMaxTok = 64;                   // tokens per chunk of a helper CTA (eight tiles)
constexpr int kHB = 3;                         // tile-slice buffers (steps in flight); token buffers

struct HParams {
    CUtensorMap tmap_x;      // x (fused: x_prev) as (hc, d/hc, s, T), box (hc, hsc, s, kHT)
    CUtensorMap tmap_w;      // fn_w, box (hc, hsc, s, R)
    CUtensorMap tmap_f;      // fused: f as [T][1][d], box (hc, hsc, 1, kHT)
    CUtensorMap tmap_xnew;   // fused: x_new, boxes as for x
    const float *x, *scale, *base, *post_prev, *comb_prev;
    float *pre, *post, *comb, *y, *x_new;
    float *part;             // [tokens from t0][2 * kCS][RV]: the helper tokens' partials
    StatusBlock *status;
    int T, d, hs, hsc, LK, NJ, iters;
    int y_rows;              // rows of y (the call's T), as in Params
    int t0;                  // first helper token
    int ntiles;              // helper tiles: tile i holds tokens [t0 + kHT*i, t0 + kHT*i + kHT) below T
    float eps, invK;
};

struct HLay {
    int off_w, off_x, off_f, off_coef, off_sink, off_pre, off_bar, off_misc, total;
};

template <int S>
__host__ __device__ inline HLay make_hlay()
{
    using G = CG<S, false, 4>;
    HLay L;
    int o = 0;
    L.off_w = o;      // [RP][LK]: the fn_w slice (rows past R zero)
    o += G::RP * kMaxLK * 4;
    L.off_x = o;      // [kHB][kHT][LK]: tile slices in flight
    o += kHB * kHT * kMaxLK * 4;
    L.off_f = o;      // [kHB][kHT][hs]: fused, their f slices
    o += kHB * kHT * kMaxFusedHs * 4;
    // Phase 2 lays kHB token slabs (s*d <= 16 * kMaxLK floats each) over all of the above.
    o = o > kHB * 16 * kMaxLK * 4 ? o : kHB * 16 * kMaxLK * 4;
    L.off_coef = o;   // [kHMaxTok][s + s*s]: fused, post/comb of the CTA's tokens
    o += kHMaxTok * (S + S * S) * 4;
    L.off_sink = o;   // [kHMaxTok][16]: exp(comb logits)
    o += kHMaxTok * 16 * 4;
    L.off_pre = o;    // [kHMaxTok][4]: pre gates
    o += kHMaxTok * 4 * 4;
    L.off_bar = o;    // xfull[kHB], wfull, tfull[kHB]
    o += (2 * kHB + 1) * 8;
    L.off_misc = o;   // abort flag; loads issued into each x buffer, fn_w, each token buffer; TMEM address;
    o += 64;          // the warps done with the fn_w staging buffer, with each x buffer
    L.total = o;
    return L;
}

template <int S>
__global__ void __launch_bounds__(kHThreads, 1) hc_pre_helper_kernel(const __grid_constant__ HParams p)
{
    constexpr int RG = 4, NT = kHNT;
    using G = CG<S, false, RG>;
    using C = CT<S, NT, false, RG>;
    constexpr int NC = S + S * S;
    constexpr int kHCT = kHMaxTok / kHT;   // tiles per chunk
    extern __shared__ __align__(128) unsigned char smem[];
    const HLay L = make_hlay<S>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *wsm = reinterpret_cast<float *>(smem + L.off_w);
    float *xb = reinterpret_cast<float *>(smem + L.off_x);
    float *fb = reinterpret_cast<float *>(smem + L.off_f);
    float *coef_s = reinterpret_cast<float *>(smem + L.off_coef);
    float *sink_s = reinterpret_cast<float *>(smem + L.off_sink);
    float *pre_s = reinterpret_cast<float *>(smem + L.off_pre);
    const uint32_t bar0 = ptx::smem_u32(smem + L.off_bar);
    auto XFULL = [&](int b) { return bar0 + 8u * (uint32_t)b; };
    const uint32_t WFULL = bar0 + 8u * kHB;
    auto TFULL = [&](int b) { return bar0 + 8u * (uint32_t)(kHB + 1 + b); };   // phase 2: token buffers
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);   // x [kHB], fn_w, tokens [kHB]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc + 40);
    int *rel_w = reinterpret_cast<int *>(smem + L.off_misc + 44);   // then rel_x[kHB]
    int *rel_x = rel_w + 1;
    StatusBlock *sb = p.status;
    const bool fused = p.x_new != nullptr;
    // This CTA's tiles [k0, k1), taken in chunks of at most kHCT tiles (kHMaxTok tokens):
    // chunk q, slice c, tile j of the chunk is step g = 16 kHCT q + c nq + j.
    const int k0 = (int)((long long)blockIdx.x * p.ntiles / gridDim.x);
    const int k1 = (int)((long long)(blockIdx.x + 1) * p.ntiles / gridDim.x);
    const int nmy = k1 - k0;
    const int nchunk = (nmy + kHCT - 1) / kHCT;
    auto chunk_tiles = [&](int q) { return min(kHCT, nmy - q * kHCT); };
    const int stage_floats = kHT * p.LK;
    const uint32_t xbytes = (uint32_t)(stage_floats * 4), fbytes = (uint32_t)(kHT * p.hs * 4);

    if (threadIdx.x == 0) {
        for (int b = 0; b < kHB; ++b) {
            ptx::mbar_init(XFULL(b), 1);
            ptx::mbar_init(TFULL(b), 1);
        }
        ptx::mbar_init(WFULL, 1);
        for (int i = 0; i < 2 * kHB + 1; ++i)
            issued[i] = 0;
        for (int i = 0; i < kHB + 1; ++i)
            rel_w[i] = 0;
        *abort_flag = *reinterpret_cast<volatile unsigned *>(&sb->code) != 0u ? 2 : 0;
        ptx::fence_mbar_init_cluster();
    }
    if (warp == 0) {   // the fn_w slice in use lives in TMEM (the CTA is alone on its SM)
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tmem_fence_before_sync();
    __syncthreads();
    ptx::tmem_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const bool skip = *abort_flag == 2 || nmy <= 0;

    auto issue = [&](int g) {   // one thread: step g's tile slice (and f slice) into buffer g % kHB
        const int q = g / (kCS * kHCT), r = g - q * kCS * kHCT, nq = chunk_tiles(q);
        const int c = r / nq, j = r - c * nq, b = g % kHB;
        const int t0 = p.t0 + (k0 + q * kHCT + j) * kHT;
        ptx::mbar_arrive_expect_tx(XFULL(b), xbytes + (fused ? fbytes : 0u));
        ptx::tma_load_4d(ptx::smem_u32(xb + b * stage_floats), &p.tmap_x, 0, c * p.hsc, 0, t0, XFULL(b));
        if (fused)
            ptx::tma_load_4d(ptx::smem_u32(fb + b * kHT * kMaxFusedHs), &p.tmap_f, 0, c * p.hsc, 0, t0, XFULL(b));
        issued[b] = issued[b] + 1;
    };
    auto load_w = [&](int c) {   // one thread: fn_w slice c
        ptx::mbar_arrive_expect_tx(WFULL, (uint32_t)(G::R * p.LK * 4));
        ptx::tma_load_4d(ptx::smem_u32(wsm), &p.tmap_w, 0, c * p.hsc, 0, 0, WFULL);
        issued[kHB] = issued[kHB] + 1;
        ptx::tma_prefetch_l2_4d(&p.tmap_w, 0, ((c + 1) % kCS) * p.hsc, 0, 0);   // the next slice into L2
    };

    bool ok = !skip;
    if (ok && threadIdx.x == 0) {
        ptx::prefetch_tmap(&p.tmap_x);
        ptx::prefetch_tmap(&p.tmap_w);
    }
    const int tg = lane >> 4, kg = lane & 15;
    const int rg = warp & 3, half = warp >> 2;
    const int njh = (p.NJ + 1) / 2;
    const int j0 = half * njh, nj = half ? p.NJ - njh : njh;
    const int lk4 = p.LK * 4;
    const int slot0 = tg * NT;
    const uint32_t trow = tmem_base + ((uint32_t)(32 * rg) << 16);   // this sub-partition's lanes
    const int tcol0 = half * (kMaxLK / 128) * G::WQ;                    // this column half's columns
    const int h4n = p.hs / 4;
    const int grp = lane < S ? 0 : (lane < 2 * S ? 1 : 2);
    const float my_scale = lane < G::R ? p.scale[grp] : 0.f;
    const float my_base = lane < G::R ? p.base[lane] : 0.f;
    int tl = 0;   // phase 2's token loads so far (token buffer tl % 2, phase tl / 2)
    for (int q = 0; ok && q < nchunk; ++q) {
        const int nq = chunk_tiles(q);
        const int tok0 = p.t0 + (k0 + q * kHCT) * kHT;   // the chunk's first token
        const int ntok = min(p.T, tok0 + nq * kHT) - tok0;
        const int g0 = kCS * kHCT * q, g1 = g0 + kCS * nq;   // the chunk's steps
        if (threadIdx.x == 0) {   // fn_w slice 0 and the first kHB steps (phase 2 of the last
            load_w(0);            // chunk is done with the buffers)
            for (int g = g0; g < g0 + kHB && g < g1; ++g)
                issue(g);
        }
        if (fused) {   // the chunk's post/comb (the previous chunk is done with the buffer)
            for (int e = threadIdx.x; e < ntok * NC; e += kHThreads) {
                const int tt = e / NC, cc = e - tt * NC;
                coef_s[e] = cc < S ? __ldg(p.post_prev + (size_t)(tok0 + tt) * S + cc)
                                   : __ldg(p.comb_prev + (size_t)(tok0 + tt) * S * S + (cc - S));
            }
            __syncthreads();
        }
        // ------------------------------------------------------------ phase 1: slices
        // Pre-chain mode: no CTA barrier.  Each warp waits for a buffer itself, and the last of
        // the eight warps to be done with a buffer (a shared counter) issues its next load, which
        // saves the two CTA-wide barriers a step of the plain scheme.  Fused mode:
        // the transform makes each step's tokens depend on all eight warps, so one barrier per
        // step; thread 0 then stores x', loads the next fn_w slice (step 0 of a slice: every
        // warp has copied the current one) and refills the previous step's buffer.
        for (int c = 0; c < kCS; ++c) {
            // fn_w slice c: staged in shared memory (loaded during slice c - 1), then copied into
            // this thread's TMEM lane, which only this thread reads: warp (rg, half) lane kg's
            // values of column group jj at columns half*8*WQ + jj*WQ, row r's pairs (2kg, 2kg+1)
            // and (32+2kg, 33+2kg) at 4r .. 4r+3 (rows past R zero).
            if (ok)
                ok = warp_wait<false>(lane, WFULL, c & 1, abort_flag, sb, kSiteWFull);
            if (!ok && !fused)
                break;
            if (ok) {
                for (int jj = 0; jj < nj; ++jj) {
                    const int col = 64 * (j0 + jj) + 2 * kg;
#pragma unroll
                    for (int r = 0; r < G::B; ++r) {
                        const int row = rg * G::B + r;
                        float2 v0 = make_float2(0.f, 0.f), v1 = make_float2(0.f, 0.f);
                        if (row < G::R) {
                            v0 = *reinterpret_cast<const float2 *>(wsm + row * p.LK + col);
                            v1 = *reinterpret_cast<const float2 *>(wsm + row * p.LK + col + 32);
                        }
                        const float a[4] = {v0.x, v0.y, v1.x, v1.y};
                        ptx::tmem_st4(trow + (uint32_t)(tcol0 + jj * G::WQ + 4 * r), a);
                    }
                }
                ptx::tmem_wait_st();
            }
            if (!fused) {
                __syncwarp();
                if (lane == 0) {   // the last warp out of the staging buffer refills it
                    __threadfence_block();
                    if (atomicAdd(rel_w, 1) % 8 == 7 && c + 1 < kCS) {
                        __threadfence_block();
                        load_w(c + 1);
                    }
                }
            }
            for (int j = 0; j < nq; ++j) {
                const int g = kCS * kHCT * q + c * nq + j, b = g % kHB;
                if (ok)
                    ok = warp_wait<false>(lane, XFULL(b), (g / kHB) & 1, abort_flag, sb, kSiteXFull);
                if (!ok && !fused)
                    break;
                const int t0 = tok0 + j * kHT;
                const int tm = min(kHT, p.T - t0);
                float *xs = xb + b * stage_floats;
                if (fused) {
                    // The previous site's hc_post on the slice, in place (hc_post's operations
                    // in hc_post's order): warp t owns token t of the tile, lanes its float4s.
                    const int t = warp;
                    if (ok && t < tm) {
                        float cf[NC];
#pragma unroll
                        for (int m = 0; m < NC; ++m)
                            cf[m] = coef_s[(j * kHT + t) * NC + m];
                        const float *fr = fb + b * kHT * kMaxFusedHs + t * p.hs;
                        for (int h4 = lane; h4 < h4n; h4 += 32) {
                            float4 *xt = reinterpret_cast<float4 *>(xs + t * p.LK + 4 * h4);
                            const float4 fv = *reinterpret_cast<const float4 *>(fr + 4 * h4);
                            float4 xv[S];
#pragma unroll
                            for (int m = 0; m < S; ++m)
                                xv[m] = xt[m * h4n];
#pragma unroll
                            for (int k = 0; k < S; ++k) {
                                const float pk = cf[k];
                                float4 o = make_float4(pk * fv.x, pk * fv.y, pk * fv.z, pk * fv.w);
#pragma unroll
                                for (int m = 0; m < S; ++m) {
                                    const float cc = cf[S + m * S + k];
                                    o.x = fmaf(cc, xv[m].x, o.x);
                                    o.y = fmaf(cc, xv[m].y, o.y);
                                    o.z = fmaf(cc, xv[m].z, o.z);
                                    o.w = fmaf(cc, xv[m].w, o.w);
                                }
                                xt[k * h4n] = o;
                            }
                        }
                    }
                    ptx::fence_proxy_async_smem();   // the TMA store reads the slice
                    ok = __syncthreads_and(ok ? 1 : 0) != 0;
                    if (!ok)
                        break;
                    if (threadIdx.x == 0) {
                        ptx::tma_store_4d(&p.tmap_xnew, 0, c * p.hsc, 0, t0, ptx::smem_u32(xs));
                        ptx::bulk_commit();
                        if (j == 0 && c + 1 < kCS)
                            load_w(c + 1);
                        if (g > g0 && g - 1 + kHB < g1) {   // step g - 1's buffer, once its x' is read
                            ptx::bulk_wait_read<1>();
                            issue(g - 1 + kHB);
                        }
                    }
                }
                // The decode variant's dots of slice c: warp (row group rg, column half),
                // half-warp tg on token slots [4 tg, 4 tg + 4), lane kg a K-group.
                const int ntok_h = min(NT, max(0, tm - slot0));
                const uint32_t xs_addr = ptx::smem_u32(xs + slot0 * p.LK) + 8u * kg;
                float2 acc[NT][G::B];
                float2 ssa[C::NSS];
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int r = 0; r < G::B; ++r)
                        acc[i][r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int m = 0; m < C::NSS; ++m)
                    ssa[m] = make_float2(0.f, 0.f);
                for (int jj = 0; jj < nj; ++jj) {
                    const uint32_t cofs = 256u * (uint32_t)(j0 + jj);
                    float w[G::WQ];   // the values the decode variant reads from its shared copy
                    ptx::tmem_ld_issue<G::WQ>(trow + (uint32_t)(tcol0 + jj * G::WQ), w);
                    ptx::tmem_ld_wait_regs<G::WQ>(w);
                    dots_step_smem<G::B, NT, RG, C::NSS>(acc, ssa, w, xs_addr, cofs, lk4, rg);
                }
                float v[C::NVP];
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int r = 0; r < G::B; ++r)
                        v[i * G::B + r] = acc[i][r].x + acc[i][r].y;
#pragma unroll
                for (int m = 0; m < C::NSS; ++m)
                    v[NT * G::B + m] = ssa[m].x + ssa[m].y;
#pragma unroll
                for (int m = C::NV; m < C::NVP; ++m)
                    v[m] = 0.f;
                reduce_scatter16<C::NVP>(v, kg);
                // Partials of (token, slice c, column half), in the cluster kernel's
                // receive layout.
#pragma unroll
                for (int m = 0; m < C::VPL; ++m) {
                    const int o = C::VPL * kg + m;
                    int i = NT, vid = -1;
                    if (o < NT * G::B) {
                        i = o / G::B;
                        const int row = rg * G::B + (o - i * G::B);
                        vid = row < G::R ? row : -1;
                    } else if (o < C::NV) {
                        i = rg + RG * (o - NT * G::B);
                        vid = G::R;
                    }
                    if (vid >= 0 && i < ntok_h) {
                        const int tr = t0 + slot0 + i - p.t0;
                        store_checked(p.part, ((size_t)tr * 2 * kCS + 2 * c + half) * G::RV + vid,
                                      (size_t)(p.T - p.t0) * 2 * kCS * G::RV, v[m], p.status, kStorePart);
                    }
                }
                if (!fused) {
                    __syncwarp();
                    if (lane == 0) {   // the last warp out of buffer b refills it
                        __threadfence_block();
                        if (atomicAdd(rel_x + b, 1) % 8 == 7 && g + kHB < g1) {
                            __threadfence_block();
                            issue(g + kHB);
                        }
                    }
                }
            }
            if (!ok)
                break;
        }
        // ------------------------------------------------------------ phase 2: the chunk's tokens
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        if (!ok)
            break;
        // y comes from each token's whole slab of x (fused: x', as stored above; s*d floats,
        // contiguous, at most 64 KiB), one bulk copy per token into kHB buffers laid over the
        // fn_w staging buffer and the tile-slice buffers, which phase 1 no longer needs.  The
        // first copies start now, under the gates and the Sinkhorn.
        const float *xsrc = fused ? p.x_new : p.x;
        const int d4 = p.d / 4;
        const uint32_t slab_bytes = (uint32_t)(S * p.d * 4);
        float *tbuf = wsm;
        const int tlb = tl;   // token i of the chunk is the (tlb + i)-th token load
        auto load_token = [&](int i) {   // one thread
            const int b = (tlb + i) % kHB;
            ptx::mbar_arrive_expect_tx(TFULL(b), slab_bytes);
            ptx::bulk_g2s(ptx::smem_u32(tbuf + (size_t)b * (16 * kMaxLK)), xsrc + (size_t)(tok0 + i) * S * p.d,
                          slab_bytes, TFULL(b));
            issued[kHB + 1 + b] = issued[kHB + 1 + b] + 1;
        };
        if (threadIdx.x == 0) {
            if (fused) {
                ptx::bulk_wait_all();   // the chunk's x' slices are in memory before they are read back
                ptx::fence_proxy_async_global();
            }
            for (int i = 0; i < kHB && i < ntok; ++i)
                load_token(i);
        }
        for (int i = warp; i < ntok; i += kHThreads / 32) {   // gates: one warp per token
            const int tr = tok0 + i - p.t0;
            float val = 0.f;
            if (lane <= G::R) {
                float src[2 * kCS];
#pragma unroll
                for (int m = 0; m < 2 * kCS; ++m)
                    src[m] = p.part[((size_t)tr * 2 * kCS + m) * G::RV + lane];
                val = tree_sum<2 * kCS>(src);   // the finisher's fixed order
            }
            const float ss = __shfl_sync(kFull, val, G::R);
            const float rinv = rsqrtf(ss * p.invK + p.eps);
            const float logit = lane < G::R ? val * rinv * my_scale + my_base : 0.f;
            const float sg = __fdividef(1.f, 1.f + __expf(-logit));
            const size_t tok = (size_t)tok0 + i;
            if (lane < S) {
                const float pre_v = sg + p.eps;
                store_checked(p.pre, tok * S + lane, (size_t)p.T * S, pre_v, p.status, kStorePre);
                pre_s[i * 4 + lane] = pre_v;
            } else if (lane < 2 * S) {
                store_checked(p.post, tok * S + (lane - S), (size_t)p.T * S, 2.f * sg, p.status, kStorePost);
            } else if (lane < G::R) {
                sink_s[i * 16 + (lane - 2 * S)] = __expf(logit);
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < ntok; i += kHThreads) {   // Sinkhorn: one token per thread
            float cm[S * S];
#pragma unroll
            for (int m = 0; m < S * S; ++m)
                cm[m] = sink_s[i * 16 + m];
            sinkhorn_regs<S>(cm, p.iters, p.eps);
#pragma unroll
            for (int m = 0; m < S * S; ++m)
                store_checked(p.comb, (size_t)(tok0 + i) * S * S + m, (size_t)p.T * S * S, cm[m], p.status, kStoreComb);
        }
        for (int i = 0; ok && i < ntok; ++i, ++tl) {   // y, in the collapse's order
            const int b = tl % kHB;
            ok = __syncthreads_and(threadIdx.x != 0 ||
                                   wait_bar<false>(TFULL(b), (tl / kHB) & 1, abort_flag, sb, kSiteXFull)) != 0;
            if (!ok)
                break;
            const float4 *xs4 = reinterpret_cast<const float4 *>(tbuf + (size_t)b * (16 * kMaxLK));
            const float4 pv = *reinterpret_cast<const float4 *>(pre_s + i * 4);
            const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
            const size_t y4 = (size_t)(tok0 + i) * p.d / 4;   // y row, float4s
            for (int e = threadIdx.x; e < d4; e += kHThreads) {
                float4 xv[S];
#pragma unroll
                for (int k = 0; k < S; ++k)
                    xv[k] = xs4[k * d4 + e];
                float4 a = make_float4(pr[0] * xv[0].x, pr[0] * xv[0].y, pr[0] * xv[0].z, pr[0] * xv[0].w);
#pragma unroll
                for (int k = 1; k < S; ++k) {
                    a.x = fmaf(pr[k], xv[k].x, a.x);
                    a.y = fmaf(pr[k], xv[k].y, a.y);
                    a.z = fmaf(pr[k], xv[k].z, a.z);
                    a.w = fmaf(pr[k], xv[k].w, a.w);
                }
                store_checked(reinterpret_cast<float4 *>(p.y), y4 + e, (size_t)p.y_rows * p.d / 4, a, p.status, kStoreY);
            }
            __syncthreads();   // buffer b is free
            if (threadIdx.x == 0 && i + kHB < ntok)
                load_token(i + kHB);
        }
        __syncthreads();   // the buffers, pre_s / sink_s / coef_s are free for the next chunk
    }
    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (threadIdx.x == 0 && !skip) {   // every load this CTA issued lands before it exits
        for (int b = 0; b < kHB; ++b) {
            if (issued[b] > 0)
                wait_bar<false>(XFULL(b), (issued[b] - 1) & 1, abort_flag, sb, kSiteDrain, false);
            if (issued[kHB + 1 + b] > 0)
                wait_bar<false>(TFULL(b), (issued[kHB + 1 + b] - 1) & 1, abort_flag, sb, kSiteDrain, false);
        }
        if (issued[kHB] > 0)
            wait_bar<false>(WFULL, (issued[kHB] - 1) & 1, abort_flag, sb, kSiteDrain, false);
        if (fused)
            ptx::bulk_wait_all();
    }
    ptx::tmem_fence_before_sync();
    __syncthreads();
    ptx::tmem_fence_after_sync();
    if (warp == 0)
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    ptx::griddep_wait();   // the cluster kernel has completed
}

// ---------------------------------------------------------------------- host side

struct VariantInfo {
    unsigned long long ctx = 0;   // context the attributes were set in (0: not yet)
    int max_clusters = 0;
};

template <int S, bool PERSIST, int NT, bool HEAD>
int max_clusters_for(int device)
{
    static std::mutex mu;
    static VariantInfo info[64];
    if (device < 0 || device >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    VariantInfo &vi = info[device];
    const unsigned long long ctx = context_id();
    if (ctx == 0 || vi.ctx != ctx) {
        // Function attributes belong to the context: set them again in a new one.
        vi.ctx = ctx;
        vi.max_clusters = 0;
        const Lay L = make_lay<S, PERSIST, HEAD>(kMaxLK);
        auto kern = hc_pre_cluster_kernel<S, PERSIST, NT, HEAD>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            cudaGetLastError();
            vi.ctx = 0;
            return 0;
        }
        vi.ctx = context_id();
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = kCS;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(kCS * 64);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = L.total;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        vi.max_clusters = n;
    }
    return vi.max_clusters;
}

template <int S, bool PERSIST, int NT, bool HEAD>
cudaError_t launch_variant(const Params &p, int nclusters, cudaStream_t st)
{
    // A persistent CTA allocates all 512 TMEM columns, so it must be alone on its
    // SM: reserve the largest shared-memory footprint whatever the shape.
    const Lay L = make_lay<S, PERSIST, HEAD>(PERSIST ? kMaxLK : p.LK);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(nclusters * kCS));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hc_pre_cluster_kernel<S, PERSIST, NT, HEAD>, p);
}

template <int S, bool HEAD>
bool supported_s(int device)
{
    return max_clusters_for<S, true, 4, HEAD>(device) > 0 && max_clusters_for<S, false, 1, HEAD>(device) > 0 &&
           max_clusters_for<S, false, 2, HEAD>(device) > 0 && max_clusters_for<S, false, 4, HEAD>(device) > 0 &&
           max_clusters_for<S, false, 8, HEAD>(device) > 0;
}

// The previous site's hc_post inputs and output, for the fused post -> pre mode.
struct FusedPost {
    const float *f, *post_prev, *comb_prev;
    float *x_new;
};

// The branch-input norm's inputs and outputs (pre-chain mode).
struct NormOut {
    const float *norm_w;
    float eps_norm;
    float *z;
    signed char *q;
    float *q_scale;
};

// Chunks per slice row: the fewest hsc with hs/hsc <= 256 floats, a multiple of 4.
int slice_chunks(int hs)
{
    for (int n = (hs + 255) / 256; n <= hs / 4; ++n)
        if (hs % n == 0 && (hs / n) % 4 == 0)
            return n;
    return 0;
}

// Map a row-major [rows][s][d] float tensor as (hc, d/hc, s, rows), hc = hs/hsc, with
// a box of (hc, hsc, s, box_rows); reads past the last row are zero-filled.
bool encode_slab_map(CUtensorMap *m, const float *base, int rows, int s, int d, int hs, int hsc, int box_rows)
{
    if (hsc < 1)
        return false;
    const int hc = hs / hsc;
    const cuuint64_t dims[4] = {(cuuint64_t)hc, (cuuint64_t)(d / hc), (cuuint64_t)s, (cuuint64_t)rows};
    const cuuint64_t strides[3] = {(cuuint64_t)hc * 4, (cuuint64_t)d * 4, (cuuint64_t)s * d * 4};   // bytes
    const cuuint32_t box[4] = {(cuuint32_t)hc, (cuuint32_t)hsc, (cuuint32_t)s, (cuuint32_t)box_rows};
    return tensor_map_f32(m, 4, base, dims, strides, box);
}

// The helper kernel's partials: [tokens][2 * kCS][RV] floats after the status block (and
// the stamps of a phase-stamp build).
size_t helper_part_bytes(int ntok, int s)
{
    const int rv = ((2 + s) * s + 1 + 3) / 4 * 4;
    return (size_t)ntok * 2 * kCS * (size_t)rv * 4;
}

// How many 8-token tiles the helper takes from the end of a batch of T tokens: the split
// that evens out the two kernels' times in a model fitted to GB300 timings at d = 4096,
// s = 4 (a 16-token tile per cluster every pm µs after fm µs; an 8-token tile per helper CTA
// every ph µs, plus fh µs a chunk of kHMaxTok tokens for its first fn_w slice and its second
// phase).  The cluster kernel keeps a multiple of 16 tokens and at least one tile per cluster.
// (Exposed through hc_pre_helper_tokens.)
struct HelperPlan {
    int t_main = 0;   // tokens [0, t_main) for the cluster kernel
    int ntiles = 0;   // helper tiles from t_main (0: no helper)
    int nh = 0;       // helper CTAs
};

HelperPlan plan_helper(int T, int nc, int sm_count, bool fused)
{
    HelperPlan hp;
    hp.t_main = T;
    const int nh = sm_count - kCS * nc;
    if (nh < 1 || nc < 1)
        return hp;
    const double pm = fused ? 4.39 : 3.56, fm = 8.0, ph = fused ? 46.0 : 37.0, fh = fused ? 29.0 : 26.0;
    auto main_us = [&](int tm) { return std::ceil((double)((tm + kTMT - 1) / kTMT) / nc) * pm + fm; };
    double best = main_us(T);
    for (int k = 1;; ++k) {
        const int tm = (T - k * nh * kHT + kTMT - 1) / kTMT * kTMT;   // helper: at most k tiles a CTA
        if (tm < kTMT * nc)
            break;
        const int htiles = (T - tm + kHT - 1) / kHT;
        const int per = (htiles + nh - 1) / nh;
        const double t = std::max(main_us(tm), per * ph + fh * ((per + kHMaxTok / kHT - 1) / (kHMaxTok / kHT)));
        if (t < best) {
            best = t;
            hp.t_main = tm;
            hp.ntiles = htiles;
            hp.nh = nh;
        }
    }
    return hp;
}

struct HelperInfo {
    unsigned long long ctx = 0;
    bool ok = false;
};

template <int S>
bool helper_ready(int device)
{
    static std::mutex mu;
    static HelperInfo info[64];
    if (device < 0 || device >= 64)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    HelperInfo &hi = info[device];
    const unsigned long long ctx = context_id();
    if (ctx == 0 || hi.ctx != ctx) {
        hi.ok = cudaFuncSetAttribute(hc_pre_helper_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     make_hlay<S>().total) == cudaSuccess;
        if (!hi.ok)
            cudaGetLastError();
        hi.ctx = hi.ok ? context_id() : 0;
    }
    return hi.ok;
}

// The split for a prefill batch on `device` (no helper if its kernel cannot be set up there
// or the workspace cannot hold its partials).
template <int S>
HelperPlan helper_plan_for(int T, int device, bool fused, size_t ws_bytes, int nc_persist)
{
    DeviceInfo di;
    if (!device_info(di) || !helper_ready<S>(device))
        return HelperPlan();
    HelperPlan hp = plan_helper(T, nc_persist, di.sm_count, fused);
    if (hp.ntiles > 0 && ws_bytes < kStatusBytes + kWorkspaceExtra + helper_part_bytes(T - hp.t_main, S))
        hp = HelperPlan();
    return hp;
}

// Launch the helper kernel behind the cluster kernel just queued on `st` (its parameters
// p, whose T is already the cluster kernel's share) for the batch's tokens [hp.t_main, T).
template <int S>
cudaError_t launch_helper(const Params &p, const HelperPlan &hp, int T, void *workspace, cudaStream_t st)
{
    HParams h = {};
    const bool fused = p.x_new != nullptr;
    if (!encode_slab_map(&h.tmap_x, p.x, T, S, p.d, p.hs, p.hsc, kHT))
        return cudaErrorInvalidValue;
    h.tmap_w = p.tmap_w;
    if (fused && (!encode_slab_map(&h.tmap_f, p.f, T, 1, p.d, p.hs, p.hsc, kHT) ||
                  !encode_slab_map(&h.tmap_xnew, p.x_new, T, S, p.d, p.hs, p.hsc, kHT)))
        return cudaErrorInvalidValue;
    h.x = p.x;
    h.scale = p.scale;
    h.base = p.base;
    h.post_prev = p.post_prev;
    h.comb_prev = p.comb_prev;
    h.pre = p.pre;
    h.post = p.post;
    h.comb = p.comb;
    h.y = p.y;
    h.x_new = p.x_new;
    h.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + kStatusBytes + kWorkspaceExtra);
    h.status = p.status;
    h.T = T;
    h.y_rows = p.y_rows;
    h.d = p.d;
    h.hs = p.hs;
    h.hsc = p.hsc;
    h.LK = p.LK;
    h.NJ = p.NJ;
    h.iters = p.iters;
    h.t0 = hp.t_main;
    h.ntiles = hp.ntiles;
    h.eps = p.eps;
    h.invK = p.invK;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)hp.nh);
    cfg.blockDim = dim3(kHThreads);
    cfg.dynamicSmemBytes = (size_t)make_hlay<S>().total;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, hc_pre_helper_kernel<S>, h);
}

template <int S, bool HEAD>
cudaError_t run_s(const float *x, const float *fn_w, const float *scale, const float *base, int T,
                  int d, int iters, float eps, float *pre, float *post, float *comb, float *y,
                  void *workspace, cudaStream_t st, int device, const FusedPost *fp = nullptr,
                  const NormOut *no = nullptr, size_t ws_bytes = 0)
{
    Params p = {};
    if (no) {
        p.norm_w = no->norm_w;
        p.eps_norm = no->eps_norm;
        p.z = no->z;
        p.q = no->q;
        p.q_scale = no->q_scale;
        p.inv_d = 1.0f / (float)d;
    }
    if (fp) {
        p.f = fp->f;
        p.post_prev = fp->post_prev;
        p.comb_prev = fp->comb_prev;
        p.x_new = fp->x_new;
    }
    p.x = x;
    p.fn_w = fn_w;
    p.scale = scale;
    p.base = base;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.status = static_cast<StatusBlock *>(workspace);
#ifdef HC_STAMPS
    p.stamps = reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + kStatusBytes);
#endif
    p.T = T;
    p.d = d;
    p.hs = d / kCS;
    p.hsc = slice_chunks(p.hs);
    p.LK = S * p.hs;
    p.NJ = p.LK / 64;
    p.iters = iters;
    p.eps = eps;
    p.invK = 1.0f / (float)(S * d);
    p.y_rows = T;
#ifdef HC_DEBUG_BOUNDS
    // Bounds-checked build only: pretend y has fewer rows, so that the checks' report can be
    // tested (the stores they refuse are inside the real buffer).
    if (const char *e = getenv("HC_DEBUG_BOUNDS_Y_ROWS"))
        p.y_rows = atoi(e);
#endif
    // Every decode instantiation has the same footprint; NT = 8 bounds the others.
    const int nc_decode = max_clusters_for<S, false, 8, HEAD>(device);
    const int nc_persist = max_clusters_for<S, true, 4, HEAD>(device);
    if (nc_decode < 1 || nc_persist < 1)
        return cudaErrorNotSupported;
    const bool decode = T <= nc_decode * kTMT;
    // Decode: one tile per cluster, tokens spread over as many clusters as can run
    // at once; prefill: 16-token tiles on persistent clusters.
    p.tm_tile = decode ? (T + nc_decode - 1) / nc_decode : kTMT;
    p.ntiles = (T + p.tm_tile - 1) / p.tm_tile;
    if (p.x_new && (!encode_slab_map(&p.tmap_f, p.f, T, 1, d, p.hs, p.hsc, p.tm_tile) ||
                    !encode_slab_map(&p.tmap_xnew, p.x_new, T, S, d, p.hs, p.hsc, p.tm_tile)))
        return cudaErrorInvalidValue;
    if (!encode_slab_map(&p.tmap_x, x, T, S, d, p.hs, p.hsc, p.tm_tile) ||
        !encode_slab_map(&p.tmap_w, fn_w, CG<S, HEAD>::R, S, d, p.hs, p.hsc, CG<S, HEAD>::R))
        return cudaErrorInvalidValue;
    if (decode) {
        // The token-slot count is the smallest that holds a tile.
        if (p.tm_tile <= 2)
            return launch_variant<S, false, 1, HEAD>(p, p.ntiles, st);
        if (p.tm_tile <= 4)
            return launch_variant<S, false, 2, HEAD>(p, p.ntiles, st);
        if (p.tm_tile <= 8)
            return launch_variant<S, false, 4, HEAD>(p, p.ntiles, st);
        return launch_variant<S, false, 8, HEAD>(p, p.ntiles, st);
    }
    // Prefill: the persistent clusters, and on the SMs they leave free the helper kernel for
    // the batch's last tokens (pre-chain and fused modes, when the workspace holds its partials).
    const HelperPlan hp = (!HEAD && !no) ? helper_plan_for<S>(T, device, p.x_new != nullptr, ws_bytes, nc_persist)
                                         : HelperPlan();
    if (hp.ntiles > 0) {
        p.T = hp.t_main;
        p.ntiles = hp.t_main / kTMT;
    }
    const cudaError_t e = launch_variant<S, true, 4, HEAD>(p, min(p.ntiles, nc_persist), st);
    if (e != cudaSuccess || hp.ntiles == 0)
        return e;
    return launch_helper<S>(p, hp, T, workspace, st);
}

}  // namespace

bool cluster_shape_ok(int s, int d)
{
    if (s < 1 || s > 4 || d % (kCS * 4) != 0)
        return false;
    const int LK = s * (d / kCS);
    return LK % 64 == 0 && LK <= kMaxLK && slice_chunks(d / kCS) > 0;
}

bool cluster_supported(int s, int d, bool head)
{
    if (!cluster_shape_ok(s, d))
        return false;
    DeviceInfo di;
    if (!device_info(di) || di.cc_major != 10)
        return false;
    switch (s) {
    case 1: return head ? supported_s<1, true>(di.device) : supported_s<1, false>(di.device);
    case 2: return head ? supported_s<2, true>(di.device) : supported_s<2, false>(di.device);
    case 3: return head ? supported_s<3, true>(di.device) : supported_s<3, false>(di.device);
    case 4: return head ? supported_s<4, true>(di.device) : supported_s<4, false>(di.device);
    default: return false;
    }
}

bool cluster_supported(int s, int d) { return cluster_supported(s, d, false); }

bool cluster_fused_supported(int s, int d) { return d / kCS <= kMaxFusedHs && cluster_supported(s, d, false); }

cudaError_t launch_pre_cluster(const float *x, const float *fn_w, const float *scale,
                               const float *base, int T, int s, int d, int iters, float eps,
                               float *pre, float *post, float *comb, float *y, void *workspace,
                               size_t ws_bytes, cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    switch (s) {
#define HC_CASE(S)                                                                                  \
    case S:                                                                                         \
        return run_s<S, false>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, \
                               di.device, nullptr, nullptr, ws_bytes);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4)
#undef HC_CASE
    default: return cudaErrorInvalidValue;
    }
}

int cluster_helper_tokens(int T, int s, int d, bool fused, size_t ws_bytes)
{
    if (!cluster_supported(s, d, false) || (fused && !cluster_fused_supported(s, d)))
        return 0;
    DeviceInfo di;
    if (!device_info(di))
        return 0;
    auto tokens = [&](int nc_decode, int nc_persist, HelperPlan (*plan)(int, int, bool, size_t, int)) {
        if (nc_decode < 1 || nc_persist < 1 || T <= nc_decode * kTMT)
            return 0;
        const HelperPlan hp = plan(T, di.device, fused, ws_bytes, nc_persist);
        return hp.ntiles > 0 ? T - hp.t_main : 0;
    };
    switch (s) {
#define HC_CASE(S)                                                                                  \
    case S:                                                                                         \
        return tokens(max_clusters_for<S, false, 8, false>(di.device), max_clusters_for<S, true, 4, false>(di.device), \
                      helper_plan_for<S>);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4)
#undef HC_CASE
    default: return 0;
    }
}

size_t cluster_helper_workspace_bytes(int T, int s, int d)
{
    if (T <= 0 || !cluster_shape_ok(s, d))
        return 0;
    return kStatusBytes + kWorkspaceExtra + helper_part_bytes(T, s);
}

bool cluster_norm_supported(int s, int d) { return (d / kCS) % 32 == 0 && cluster_supported(s, d, false); }

int cluster_decode_tokens(int s, int d)
{
    DeviceInfo di;
    if (!cluster_norm_supported(s, d) || !device_info(di))
        return 0;
    int nc = 0;
    switch (s) {
    case 1: nc = max_clusters_for<1, false, 8, false>(di.device); break;
    case 2: nc = max_clusters_for<2, false, 8, false>(di.device); break;
    case 3: nc = max_clusters_for<3, false, 8, false>(di.device); break;
    case 4: nc = max_clusters_for<4, false, 8, false>(di.device); break;
    default: return 0;
    }
    return nc * kTMT;
}

cudaError_t launch_pre_norm_cluster(const float *x, const float *fn_w, const float *scale,
                                    const float *base, int T, int s, int d, int iters, float eps,
                                    const float *norm_w, float eps_norm, float *pre, float *post, float *comb,
                                    float *y, float *z, signed char *q, float *q_scale, void *workspace,
                                    cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    const NormOut no{norm_w, eps_norm, z, q, q_scale};
    switch (s) {
#define HC_CASE(S)                                                                                  \
    case S:                                                                                         \
        return run_s<S, false>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, \
                               di.device, nullptr, &no);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4)
#undef HC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_post_pre_cluster(const float *x_prev, const float *f, const float *post_prev,
                                    const float *comb_prev, const float *fn_w, const float *scale,
                                    const float *base, int T, int s, int d, int iters, float eps,
                                    float *x_new, float *pre, float *post, float *comb, float *y,
                                    void *workspace, size_t ws_bytes, cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    const FusedPost fp{f, post_prev, comb_prev, x_new};
    switch (s) {
#define HC_CASE(S)                                                                                  \
    case S:                                                                                         \
        return run_s<S, false>(x_prev, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, \
                               st, di.device, &fp, nullptr, ws_bytes);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4)
#undef HC_CASE
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_head_cluster(const float *x, const float *fn_w, const float *scale,
                                const float *base, int T, int s, int d, float eps, float *gates,
                                float *y, void *workspace, cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    switch (s) {
#define HC_CASE(S)                                                                                  \
    case S:                                                                                         \
        return run_s<S, true>(x, fn_w, scale, base, T, d, 1, eps, gates, nullptr, nullptr, y, workspace, \
                              st, di.device);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4)
#undef HC_CASE
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace hc
