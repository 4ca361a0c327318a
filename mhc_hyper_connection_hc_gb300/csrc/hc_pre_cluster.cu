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
//  * Each token tile (<= 16 tokens) is brought in by bulk copies (the TMA
//    engine) into a shared-memory stage and stays there until its collapse, so
//    x is read from HBM exactly once.
//  * The fn_w slice stays resident in the CTA for every tile it processes: in
//    tensor memory (TMEM, tcgen05.ld into registers) for the persistent prefill
//    variant, in shared memory for the one-tile decode variant.  It is read
//    from L2/HBM once per CTA.
//  * Four compute warps (one per TMEM sub-partition) each own R/4 rows; in a
//    warp, lanes 0-15 take tile tokens 0-7 and lanes 16-31 tokens 8-15, and
//    lane&15 is the K-group owning float4 columns kg, kg+16, ... of the slice.
//    Per float4 column group a thread does 8 tokens x B rows x 4 FMAs (CUDA
//    cores, float32, no TF32: the 24-row contraction is too skinny for tensor
//    cores to pay and must stay in f32).
//  * The 16 K-groups are summed by an xor reduce-scatter inside each
//    half-warp, and every CTA pushes its partial dots and sum of squares for
//    token t to CTA t (the token's owner) through distributed shared memory.
//  * Two finisher warps (even/odd tiles) of each owner sum the 16 partials in
//    rank order, apply the rsqrt rescale, form the gates, broadcast pre to all
//    16 CTAs, and run the Sinkhorn in registers while the compute warps
//    already work on the next tile.  Compute warps collapse tile i after the
//    dots of tile i+1, so the exchange latency is hidden.
//  * Every wait on an mbarrier is bounded (2 s of %globaltimer); on timeout the
//    kernel records the site in the workspace status word, stops issuing work,
//    lets its bulk copies land, meets the other CTAs at the final cluster
//    barrier, frees TMEM and returns.
//
// Determinism: every sum has a fixed order independent of T, of the tile a
// token lands in and of the variant, so a token's outputs are the same bits
// whatever batch it is in.
#include "hc_internal.cuh"
#include "hc_ptx.cuh"

#include <mutex>

namespace hc {
namespace {

constexpr int kCS = 16;              // CTAs per cluster (non-portable cluster size)
constexpr int kTMT = 16;             // max tokens per tile = one owner CTA per token
constexpr int kNCW = 8;              // compute warps: two per SM sub-partition
constexpr int kProducerWarp = 8;
constexpr int kFinisherWarp = 9;     // warps 9 and 10 take even and odd tiles
constexpr int kThreads = 11 * 32;
constexpr int kComputeThreads = kNCW * 32;
constexpr int kNstPersist = 3;
constexpr int kMaxLK = 1024;         // s*d/16 <= 1024: three 64 KiB stages fit in shared memory
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr unsigned kFull = 0xffffffffu;

// mbarrier slots
constexpr int kBarXFull = 0, kBarXEmpty = 3, kBarRecv = 6, kBarPre = 8, kBarWFull = 10, kBarWFree = 11;
enum WaitSite : unsigned { kSiteWFull = 1, kSiteXFull, kSiteXEmpty, kSiteRecv, kSitePre, kSiteWFree, kSiteDrain };

template <int S>
struct CG {
    static constexpr int R = (2 + S) * S;
    static constexpr int RP = (R + kNCW - 1) / kNCW * kNCW;  // rows padded to the compute warps
    static constexpr int B = RP / kNCW;                        // rows per compute warp
    static constexpr int RV = (R + 1 + 3) / 4 * 4;             // exchange stride: R dots + sum of squares
    static constexpr int WQ = 4 * B;                           // fn_w floats per thread per column group
};

// NT = token slots per half-warp (a tile holds up to 2*NT tokens, one owner CTA each).
// Warp w sums the squares of slots w, w+4, ... so NSS values per thread.
template <int S, int NT>
struct CT {
    static constexpr int B = CG<S>::B;
    static constexpr int NSS = (NT + kNCW - 1) / kNCW;
    static constexpr int NV = NT * B + NSS;                    // per-thread values before the reduce-scatter
    static constexpr int NVP = (NV + 15) / 16 * 16;
    static constexpr int VPL = NVP / 16;                       // per-lane values after it
};

struct Lay {   // shared-memory layout in bytes
    int stage_bytes, nst, off_w, off_recv, off_pre, off_bar, off_misc, total;
};

template <int S, bool PERSIST>
__host__ __device__ inline Lay make_lay(int LK)
{
    using G = CG<S>;
    Lay L;
    L.stage_bytes = kTMT * LK * 4;
    L.nst = PERSIST ? kNstPersist : 1;
    int o = L.nst * L.stage_bytes;
    L.off_w = o;
    if (!PERSIST)
        o += G::RP * LK * 4;
    L.off_recv = o;
    o += 2 * kCS * G::RV * 4;
    L.off_pre = o;
    o += 2 * kTMT * 4 * 4;
    L.off_bar = o;
    o += 16 * 8;
    L.off_misc = o;
    o += 16;
    L.total = o;
    return L;
}

struct Params {
    const float *x, *fn_w, *scale, *base;
    float *pre, *post, *comb, *y;
    StatusBlock *status;
    int T, d, hs, LK, NJ, iters, tm_tile, ntiles;
    float eps, Kf;
};

// Bounded wait on an mbarrier phase.  honor_abort = false is used only to let
// this CTA's own bulk copies land before it exits.
template <bool CLUSTER_SCOPE>
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
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
// each row by (row sum + eps), then each column by (column sum + eps).  The
// reciprocal is the hardware approximation (__fdividef, within 2 ulp); the
// Sinkhorn's own error budget against the float64 oracle is 1e-4.
template <int S>
__device__ __forceinline__ void sinkhorn_regs(float *c, int iters, float eps)
{
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const float inv = __fdividef(1.0f, tree_sum<S>(c + j * S) + eps);
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
            const float inv = __fdividef(1.0f, tree_sum<S>(col) + eps);
#pragma unroll
            for (int j = 0; j < S; ++j)
                c[j * S + k] *= inv;
        }
    }
}

// One column group of the dots: 4 columns of the NT token slots of this half-warp,
// times this warp's B rows, as packed float32 FMAs (acc = (even-column sum,
// odd-column sum)); plus the sum of squares of this warp's own slot(s).
template <int S, int NT>
__device__ __forceinline__ void dots_step(float2 (&acc)[NT][CG<S>::B], float2 (&ssa)[CT<S, NT>::NSS],
                                          const float (&w)[CG<S>::WQ], uint32_t xs_addr,
                                          uint32_t xq_addr, uint32_t cofs, int lk4)
{
    constexpr int B = CG<S>::B;
    float4 xv[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i)
        xv[i] = ptx::lds128(xs_addr + (uint32_t)(i * lk4) + cofs);
    float4 xq[CT<S, NT>::NSS];
#pragma unroll
    for (int m = 0; m < CT<S, NT>::NSS; ++m)
        xq[m] = ptx::lds128(xq_addr + (uint32_t)(m * kNCW * lk4) + cofs);
    // Even-column halves first, then odd-column halves: consecutive packed FMAs
    // never depend on each other.
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int r = 0; r < B; ++r)
            acc[i][r] = ptx::ffma2(make_float2(xv[i].x, xv[i].y), make_float2(w[4 * r], w[4 * r + 1]), acc[i][r]);
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
        for (int r = 0; r < B; ++r)
            acc[i][r] = ptx::ffma2(make_float2(xv[i].z, xv[i].w), make_float2(w[4 * r + 2], w[4 * r + 3]), acc[i][r]);
#pragma unroll
    for (int m = 0; m < CT<S, NT>::NSS; ++m) {
        const float2 lo = make_float2(xq[m].x, xq[m].y), hi = make_float2(xq[m].z, xq[m].w);
        ssa[m] = ptx::ffma2(lo, lo, ssa[m]);
        ssa[m] = ptx::ffma2(hi, hi, ssa[m]);
    }
}

template <int S, bool PERSIST, int NT>
__global__ void __launch_bounds__(kThreads, 1) hc_pre_cluster_kernel(const Params p)
{
    using G = CG<S>;
    using C = CT<S, NT>;
    extern __shared__ __align__(128) unsigned char smem[];
    const Lay L = make_lay<S, PERSIST>(p.LK);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cid = (int)ptx::cluster_id_x(), ncl = (int)ptx::ncluster_x();
    float *stages = reinterpret_cast<float *>(smem);
    float *wsm = reinterpret_cast<float *>(smem + L.off_w);
    float *recv = reinterpret_cast<float *>(smem + L.off_recv);
    float *preb = reinterpret_cast<float *>(smem + L.off_pre);
    const uint32_t bar0 = ptx::smem_u32(smem + L.off_bar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L.off_misc + 4);
    StatusBlock *sb = p.status;
    const int K = S * p.d;
    const int stage_floats = L.stage_bytes / 4;
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };

    // ------------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < L.nst; ++s) {
            ptx::mbar_init(BAR(kBarXFull + s), 1);
            ptx::mbar_init(BAR(kBarXEmpty + s), 1);
        }
        for (int q = 0; q < 2; ++q) {
            ptx::mbar_init(BAR(kBarRecv + q), kCS);
            ptx::mbar_init(BAR(kBarPre + q), kCS);
        }
        ptx::mbar_init(BAR(kBarWFull), 1);
        ptx::mbar_init(BAR(kBarWFree), 1);
        *abort_flag = 0;
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
    ptx::cluster_sync_all();   // barriers initialised in every CTA before any remote arrive
    if (PERSIST)
        ptx::tmem_fence_after_sync();
    const uint32_t tmem_base = PERSIST ? *tmem_slot : 0u;

    if (warp == kProducerWarp) {
        // -------------------------------------------------------------- producer
        // Lane 0 does every wait and the warp follows its (broadcast) decision.
        const uint32_t hs_bytes = (uint32_t)p.hs * 4u;
        float *wdst = PERSIST ? stages : wsm;
        if (lane == 0)
            ptx::mbar_arrive_expect_tx(BAR(kBarWFull), (uint32_t)(G::R * S) * hs_bytes);
        __syncwarp();
        for (int e = lane; e < G::R * S; e += 32) {
            const int r = e / S, k = e - (e / S) * S;
            ptx::bulk_g2s(ptx::smem_u32(wdst + r * p.LK + k * p.hs),
                          p.fn_w + (size_t)r * K + (size_t)k * p.d + (size_t)rank * p.hs, hs_bytes,
                          BAR(kBarWFull));
        }
        bool ok = true;
        if (PERSIST) {   // the fn_w staging area is reused for x tiles once it sits in TMEM
            if (lane == 0)
                ok = wait_bar<false>(BAR(kBarWFree), 0, abort_flag, sb, kSiteWFree);
            ok = __shfl_sync(kFull, ok, 0);
        }
        int last_it[kNstPersist] = {-1, -1, -1};
        for (int it = 0; ok; ++it) {
            const int tile = cid + it * ncl;
            if (tile >= p.ntiles)
                break;
            const int s = it % L.nst, u = it / L.nst;
            if (u > 0) {
                if (lane == 0)
                    ok = wait_bar<false>(BAR(kBarXEmpty + s), (u - 1) & 1, abort_flag, sb, kSiteXEmpty);
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok)
                    break;
            }
            const int t0 = tile * p.tm_tile, tm = min(p.tm_tile, p.T - t0);
            if (lane == 0)
                ptx::mbar_arrive_expect_tx(BAR(kBarXFull + s), (uint32_t)(tm * S) * hs_bytes);
            __syncwarp();
            float *xs = stages + s * stage_floats;
            for (int e = lane; e < tm * S; e += 32) {
                const int t = e / S, k = e - (e / S) * S;
                ptx::bulk_g2s(ptx::smem_u32(xs + t * p.LK + k * p.hs),
                              p.x + ((size_t)(t0 + t) * S + k) * p.d + (size_t)rank * p.hs, hs_bytes,
                              BAR(kBarXFull + s));
            }
            last_it[s] = it;
        }
        // Every bulk copy this CTA issued lands before the CTA may exit.
        if (lane == 0) {
            wait_bar<false>(BAR(kBarWFull), 0, abort_flag, sb, kSiteDrain, false);
            for (int s = 0; s < L.nst; ++s)
                if (last_it[s] >= 0)
                    wait_bar<false>(BAR(kBarXFull + s), (last_it[s] / L.nst) & 1, abort_flag, sb,
                                    kSiteDrain, false);
        }
        __syncwarp();
    } else if (warp < kNCW) {
        // -------------------------------------------------------------- compute warps
        // Every thread polls each barrier itself (its own acquire); a named
        // barrier with an AND reduction then makes the go / give-up decision
        // identical in all four warps, so they always meet the same barriers.
        const int tg = lane >> 4, kg = lane & 15;
        // TMEM: warp w reads lanes 32*(w%4).. of its sub-partition; the two warps of a
        // sub-partition use disjoint column ranges.
        const uint32_t trow = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16) +
                              (uint32_t)((warp >> 2) * p.NJ * G::WQ);
        bool ok = ptx::named_bar_and(1, kComputeThreads,
                                     wait_bar<false>(BAR(kBarWFull), 0, abort_flag, sb, kSiteWFull));
        if (PERSIST && ok) {
            // This thread's fixed fn_w values -> its TMEM lane, column j*WQ + 4r + e.
            for (int j = 0; j < p.NJ; ++j) {
                const int c = 4 * (kg + 16 * j);
#pragma unroll
                for (int r = 0; r < G::B; ++r) {
                    const int row = warp * G::B + r;
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row < G::R)
                        v = *reinterpret_cast<const float4 *>(stages + row * p.LK + c);
                    const float a[4] = {v.x, v.y, v.z, v.w};
                    ptx::tmem_st4(trow + (uint32_t)(j * G::WQ + 4 * r), a);
                }
            }
            ptx::tmem_wait_st();
            ptx::named_bar_sync(1, kComputeThreads);
            if (threadIdx.x == 0)
                ptx::mbar_arrive(BAR(kBarWFree));
        }

        auto collapse = [&](int itc) -> bool {
            const int q = itc & 1;
            const bool got = wait_bar<true>(BAR(kBarPre + q), (itc >> 1) & 1, abort_flag, sb, kSitePre);
            if (!ptx::named_bar_and(1, kComputeThreads, got))
                return false;
            const int tile = cid + itc * ncl, t0 = tile * p.tm_tile;
            const int tm = min(p.tm_tile, p.T - t0);
            const int s = itc % L.nst;
            const float *xs = stages + s * stage_floats;
            const int h4n = p.hs / 4;
            int t = threadIdx.x / h4n, h4 = threadIdx.x - (threadIdx.x / h4n) * h4n;
            const uint32_t xs_base = ptx::smem_u32(xs);
            const uint32_t pre_base = ptx::smem_u32(preb + q * kTMT * 4);
            for (; t < tm;) {
                float pr[S];
#pragma unroll
                for (int k = 0; k < S; ++k)
                    pr[k] = ptx::lds32(pre_base + 4u * (uint32_t)(t * 4 + k));
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
                *reinterpret_cast<float4 *>(p.y + (size_t)(t0 + t) * p.d + (size_t)rank * p.hs + 4 * h4) = a;
                h4 += kComputeThreads;
                while (h4 >= h4n) {
                    h4 -= h4n;
                    ++t;
                }
            }
            ptx::named_bar_sync(1, kComputeThreads);
            if (threadIdx.x == 0)
                ptx::mbar_arrive(BAR(kBarXEmpty + s));   // stage free for the producer
            return true;
        };

        int it = 0;
        for (; ok; ++it) {
            const int tile = cid + it * ncl;
            if (tile >= p.ntiles)
                break;
            const int s = it % L.nst, u = it / L.nst;
            ok = ptx::named_bar_and(1, kComputeThreads,
                                    wait_bar<false>(BAR(kBarXFull + s), u & 1, abort_flag, sb, kSiteXFull));
            if (!ok)
                break;
            const int t0 = tile * p.tm_tile, tm = min(p.tm_tile, p.T - t0);
            const int ntok = min(NT, max(0, tm - NT * tg));
            // Byte address of token slot 0 of this half-warp, at this lane's first column group.
            const uint32_t xs_addr = ptx::smem_u32(stages + s * stage_floats + (tg * NT) * p.LK) + 16u * kg;
            const uint32_t ws_addr = ptx::smem_u32(wsm + (warp * G::B) * p.LK) + 16u * kg;
            // Slots warp, warp+4, ... of this half-warp: the ones whose squares this warp sums.
            const uint32_t xq_addr = xs_addr + (uint32_t)(warp * p.LK * 4);

            // Packed float32 FMAs: acc[i][r] holds (sum over even columns, sum over odd columns).
            // Every slot is computed (rows of a stage past the tile's last token hold stale but
            // harmless data, never pushed), so the loop has no data-dependent branch.
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

            const int lk4 = p.LK * 4;
            if (PERSIST) {
                // fn_w from TMEM, double-buffered without copies: wa holds even column
                // groups, wb odd ones; the load of the next group overlaps this one's FMAs.
                float wa[G::WQ], wb[G::WQ];
                ptx::tmem_ld_issue<G::WQ>(trow, wa);
                ptx::tmem_ld_wait_regs<G::WQ>(wa);
                for (int j = 0; j < p.NJ; j += 2) {
                    const bool odd = j + 1 < p.NJ;
                    if (odd)
                        ptx::tmem_ld_issue<G::WQ>(trow + (uint32_t)((j + 1) * G::WQ), wb);
                    dots_step<S, NT>(acc, ssa, wa, xs_addr, xq_addr, 256u * (uint32_t)j, lk4);
                    if (!odd)
                        break;
                    ptx::tmem_ld_wait_regs<G::WQ>(wb);
                    const bool next = j + 2 < p.NJ;
                    if (next)
                        ptx::tmem_ld_issue<G::WQ>(trow + (uint32_t)((j + 2) * G::WQ), wa);
                    dots_step<S, NT>(acc, ssa, wb, xs_addr, xq_addr, 256u * (uint32_t)(j + 1), lk4);
                    if (next)
                        ptx::tmem_ld_wait_regs<G::WQ>(wa);
                }
            } else {
                for (int j = 0; j < p.NJ; ++j) {
                    const uint32_t cofs = 256u * (uint32_t)j;
                    float w[G::WQ];
#pragma unroll
                    for (int r = 0; r < G::B; ++r) {
                        const float4 v = ptx::lds128(ws_addr + (uint32_t)(r * lk4) + cofs);
                        w[4 * r] = v.x;
                        w[4 * r + 1] = v.y;
                        w[4 * r + 2] = v.z;
                        w[4 * r + 3] = v.w;
                    }
                    dots_step<S, NT>(acc, ssa, w, xs_addr, xq_addr, cofs, lk4);
                }
            }

            // Half-warp sums over the 16 K-groups, then push to the owners.
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
            const int qb = it & 1;
#pragma unroll
            for (int q = 0; q < C::VPL; ++q) {
                const int o = C::VPL * kg + q;
                int i = NT, vid = -1;
                if (o < NT * G::B) {
                    i = o / G::B;
                    const int row = warp * G::B + (o - i * G::B);
                    vid = row < G::R ? row : -1;
                } else if (o < C::NV) {
                    i = warp + kNCW * (o - NT * G::B);
                    vid = G::R;
                }
                if (vid >= 0 && i < ntok) {
                    const uint32_t local = ptx::smem_u32(recv + (qb * kCS + (int)rank) * G::RV + vid);
                    ptx::st_cluster_f32(ptx::mapa(local, (uint32_t)(tg * NT + i)), v[q]);
                }
            }
            ptx::named_bar_sync(1, kComputeThreads);
            if (threadIdx.x < kCS) {
                ptx::fence_acq_rel_cluster();
                ptx::mbar_arrive_remote(ptx::mapa(BAR(kBarRecv + qb), threadIdx.x));
            }
            if (it > 0 && !(ok = collapse(it - 1)))
                break;
        }
        if (ok && it > 0)
            collapse(it - 1);
    } else {
        // -------------------------------------------------------------- finisher warps
        // Lane 0 waits; the acquire it performs, followed by __syncwarp, orders
        // the other lanes' reads of the remotely written partials after it.
        const int f = warp - kFinisherWarp;
        const int grp = lane < S ? 0 : (lane < 2 * S ? 1 : 2);
        const float my_scale = lane < G::R ? p.scale[grp] : 0.f;
        const float my_base = lane < G::R ? p.base[lane] : 0.f;
        for (int it = f;; it += 2) {
            const int tile = cid + it * ncl;
            if (tile >= p.ntiles)
                break;
            const int qb = it & 1;
            bool got = true;
            if (lane == 0)
                got = wait_bar<true>(BAR(kBarRecv + qb), (it >> 1) & 1, abort_flag, sb, kSiteRecv);
            got = __shfl_sync(kFull, got, 0);
            __syncwarp();
            if (!got)
                break;
            const int t0 = tile * p.tm_tile, tm = min(p.tm_tile, p.T - t0);
            const bool own = (int)rank < tm;
            float val = 0.f;
            if (own && lane <= G::R) {
                float part[kCS];
                const uint32_t a0 = ptx::smem_u32(recv + qb * kCS * G::RV + lane);
#pragma unroll
                for (int c = 0; c < kCS; ++c)
                    part[c] = ptx::lds32(a0 + 4u * (uint32_t)(c * G::RV));
                val = tree_sum<kCS>(part);   // sources in a fixed pairwise order
            }
            const float ss = __shfl_sync(kFull, val, G::R);
            const float rinv = rsqrtf(ss / p.Kf + p.eps);
            const float logit = lane < G::R ? val * rinv * my_scale + my_base : 0.f;
            const float sg = 1.f / (1.f + expf(-logit));
            const float pre_v = sg + p.eps;
            float pk[S];
#pragma unroll
            for (int k = 0; k < S; ++k)
                pk[k] = __shfl_sync(kFull, pre_v, k);
            if (lane < kCS) {
                if (own) {
                    const uint32_t loc = ptx::smem_u32(preb + (qb * kTMT + (int)rank) * 4);
#pragma unroll
                    for (int k = 0; k < S; ++k)
                        ptx::st_cluster_f32(ptx::mapa(loc + 4u * k, (uint32_t)lane), pk[k]);
                }
                ptx::mbar_arrive_remote(ptx::mapa(BAR(kBarPre + qb), (uint32_t)lane));
            }
            if (own) {
                const size_t tok = (size_t)t0 + rank;
                if (lane < S)
                    p.pre[tok * S + lane] = pre_v;
                else if (lane < 2 * S)
                    p.post[tok * S + (lane - S)] = 2.f * sg;
                const float e = (lane >= 2 * S && lane < G::R) ? expf(logit) : 0.f;
                float cm[S * S];
#pragma unroll
                for (int q = 0; q < S * S; ++q)
                    cm[q] = __shfl_sync(kFull, e, 2 * S + q);
                if (lane == 0) {
                    sinkhorn_regs<S>(cm, p.iters, p.eps);
#pragma unroll
                    for (int q = 0; q < S * S; ++q)
                        p.comb[tok * S * S + q] = cm[q];
                }
            }
            __syncwarp();
        }
    }

    // ------------------------------------------------------------------ teardown
    __syncwarp();
    if (PERSIST)
        ptx::tmem_fence_before_sync();
    ptx::cluster_sync_all();   // no CTA leaves while another may still write its shared memory
    if (PERSIST) {
        ptx::tmem_fence_after_sync();
        if (warp == 0)
            ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------------- host side

struct VariantInfo {
    bool init = false;
    int max_clusters = 0;
};

template <int S, bool PERSIST, int NT>
int max_clusters_for(int device)
{
    static std::mutex mu;
    static VariantInfo info[64];
    if (device < 0 || device >= 64)
        return 0;
    std::lock_guard<std::mutex> lock(mu);
    VariantInfo &vi = info[device];
    if (!vi.init) {
        vi.init = true;
        const Lay L = make_lay<S, PERSIST>(kMaxLK);
        auto kern = hc_pre_cluster_kernel<S, PERSIST, NT>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
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

template <int S, bool PERSIST, int NT>
cudaError_t launch_variant(const Params &p, int nclusters, cudaStream_t st)
{
    // A persistent CTA allocates all 512 TMEM columns, so it must be alone on its
    // SM: reserve the largest shared-memory footprint whatever the shape.
    const Lay L = make_lay<S, PERSIST>(PERSIST ? kMaxLK : p.LK);
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
    return cudaLaunchKernelEx(&cfg, hc_pre_cluster_kernel<S, PERSIST, NT>, p);
}

template <int S>
bool supported_s(int device)
{
    return max_clusters_for<S, true, 8>(device) > 0 && max_clusters_for<S, false, 1>(device) > 0 &&
           max_clusters_for<S, false, 2>(device) > 0 && max_clusters_for<S, false, 4>(device) > 0 &&
           max_clusters_for<S, false, 8>(device) > 0;
}

template <int S>
cudaError_t run_s(const float *x, const float *fn_w, const float *scale, const float *base, int T,
                  int d, int iters, float eps, float *pre, float *post, float *comb, float *y,
                  void *workspace, cudaStream_t st, int device)
{
    Params p;
    p.x = x;
    p.fn_w = fn_w;
    p.scale = scale;
    p.base = base;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.status = static_cast<StatusBlock *>(workspace);
    p.T = T;
    p.d = d;
    p.hs = d / kCS;
    p.LK = S * p.hs;
    p.NJ = p.LK / 64;
    p.iters = iters;
    p.eps = eps;
    p.Kf = (float)(S * d);
    // Every decode instantiation has the same footprint; NT = 8 bounds the others.
    const int nc_decode = max_clusters_for<S, false, 8>(device);
    const int nc_persist = max_clusters_for<S, true, 8>(device);
    if (nc_decode < 1 || nc_persist < 1)
        return cudaErrorNotSupported;
    if (T <= nc_decode * kTMT) {
        // One tile per cluster, tokens spread over as many clusters as can run at once;
        // the token-slot count is the smallest that holds a tile.
        p.tm_tile = (T + nc_decode - 1) / nc_decode;
        p.ntiles = (T + p.tm_tile - 1) / p.tm_tile;
        if (p.tm_tile <= 2)
            return launch_variant<S, false, 1>(p, p.ntiles, st);
        if (p.tm_tile <= 4)
            return launch_variant<S, false, 2>(p, p.ntiles, st);
        if (p.tm_tile <= 8)
            return launch_variant<S, false, 4>(p, p.ntiles, st);
        return launch_variant<S, false, 8>(p, p.ntiles, st);
    }
    p.tm_tile = kTMT;
    p.ntiles = (T + kTMT - 1) / kTMT;
    return launch_variant<S, true, 8>(p, min(p.ntiles, nc_persist), st);
}

}  // namespace

bool cluster_shape_ok(int s, int d)
{
    if (s < 1 || s > 4 || d % (kCS * 4) != 0)
        return false;
    const int LK = s * (d / kCS);
    return LK % 64 == 0 && LK <= kMaxLK;
}

bool cluster_supported(int s, int d)
{
    if (!cluster_shape_ok(s, d))
        return false;
    DeviceInfo di;
    if (!device_info(di) || di.cc_major != 10)
        return false;
    switch (s) {
    case 1: return supported_s<1>(di.device);
    case 2: return supported_s<2>(di.device);
    case 3: return supported_s<3>(di.device);
    case 4: return supported_s<4>(di.device);
    default: return false;
    }
}

cudaError_t launch_pre_cluster(const float *x, const float *fn_w, const float *scale,
                               const float *base, int T, int s, int d, int iters, float eps,
                               float *pre, float *post, float *comb, float *y, void *workspace,
                               cudaStream_t st)
{
    DeviceInfo di;
    if (!device_info(di))
        return cudaErrorNoDevice;
    switch (s) {
    case 1: return run_s<1>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di.device);
    case 2: return run_s<2>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di.device);
    case 3: return run_s<3>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di.device);
    case 4: return run_s<4>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, workspace, st, di.device);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace hc
