// hc_pre_generic.cu -- the generic pre-chain path: any 1 <= s <= 8, d % 4 == 0.
// The same two kernels, with HEAD set, serve the gated-head trunk exit (rows =
// streams, one scale, pre-style gates and the collapse; no post, no Sinkhorn).
//
// Two launches per site:
//   1. mixes_partial_kernel: for a tile of kTM tokens and one slice of the
//      K = s*d columns, the partial dots  sum_q fn_w[r, q] * x[t, q]  for all
//      R = (2+s)*s rows, plus the partial sum of squares  sum_q x[t, q]^2.
//      (memra-engine hyper.rs module header: "mixes = fn_w . x" and the
//      "mean(x^2)" of the rsqrt rescale, both over the whole s*d slab.)
//   2. finish_collapse_kernel: one block per token sums the K-slices in a
//      fixed order, applies rsqrt(mean + eps), forms the logits, the pre/post
//      gates and the Sinkhorn comb, then writes the collapse
//      y = sum_c pre_c * x[t, c, :] (module header "y[t, :] = ...").
//
// This path re-reads x for the collapse (from L2 when it is still resident),
// so it moves ~2x the algorithmic bytes; the cluster path in
// hc_pre_cluster.cu reads x once and is preferred where it applies.
//
// Determinism: the K split depends on (T, s, d) only, every partial is summed
// in a fixed order (lane order within a thread, an xor butterfly over the 16
// K-groups, then ascending K-slice), and no floating-point atomics are used,
// so repeated calls are bit-identical.
#include <mutex>

#include "hc_internal.cuh"

namespace hc {
namespace {

constexpr int kTM = 16;            // tokens per tile (2 token groups of 8)
constexpr int kKC = 128;           // columns per K chunk staged in shared memory
constexpr int kTargetCtas = 304;   // split-K sizing: 2 x the 152 SMs of a GB300 (the s = 4 kernel
                                   // holds 3 CTAs per SM, s >= 7 one)
constexpr int kFinishThreads = 256;

// HEAD: the gated-head trunk exit (rows = streams, pre-style gates only).
template <int S, bool HEAD = false>
struct Geo {
    static constexpr int R = HEAD ? S : (2 + S) * S;
    static constexpr int NW = R / S;             // one warp per row group of S rows
    static constexpr int NT = 32 * NW;
    static constexpr int XS = kTM * kKC;         // floats of x per stage
    static constexpr int WS = R * kKC;           // floats of fn_w per stage
    static constexpr int STAGE = XS + WS;
    static constexpr size_t SMEM = 2 * (size_t)STAGE * sizeof(float);
};

struct Split {
    int nt;       // token tiles
    int nks;      // K slices
    int nck;      // K chunks in total
    int ck_per;   // chunks per slice
};

Split make_split(int T, int s, int d)
{
    const long K = (long)s * d;
    Split sp;
    sp.nck = (int)((K + kKC - 1) / kKC);
    sp.nt = (T + kTM - 1) / kTM;
    int nks = sp.nt > 0 ? (kTargetCtas + sp.nt - 1) / sp.nt : 1;
    nks = nks < 1 ? 1 : (nks > sp.nck ? sp.nck : nks);
    sp.ck_per = (sp.nck + nks - 1) / nks;
    sp.nks = (sp.nck + sp.ck_per - 1) / sp.ck_per;   // no empty slices
    return sp;
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, int src_bytes)
{
    const unsigned dst = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(gsrc),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// Thread layout: warp w owns rows [w*S, w*S+S); in each warp, lanes 0-15 are
// token group 0 (tile tokens 0-7) and lanes 16-31 token group 1 (tokens 8-15);
// lane & 15 is the K-group, which owns float4 columns kg and kg+16 of every
// 128-column chunk.  Per chunk a thread does 2 x 8 x S x 4 FMAs from 2*(8+S)
// 128-bit shared loads; warp 0 also accumulates the sums of squares.
template <int S, bool HEAD>
__global__ void __launch_bounds__(Geo<S, HEAD>::NT)
mixes_partial_kernel(const float *__restrict__ x, const float *__restrict__ fn_w, int T, int K,
                     int nck, int ck_per, float *__restrict__ part)
{
    using G = Geo<S, HEAD>;
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const int t0 = blockIdx.x * kTM;
    const int ks = blockIdx.y;
    const int ck0 = ks * ck_per;
    const int ck1 = min(nck, ck0 + ck_per);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tg = lane >> 4, kg = lane & 15;
    const int r0 = warp * S;

    auto load_chunk = [&](int ck, int stage) {
        float *xs = sm + stage * G::STAGE;
        float *ws = xs + G::XS;
        const long q0 = (long)ck * kKC;
        for (int e = threadIdx.x; e < kTM * (kKC / 4); e += G::NT) {
            const int row = e / (kKC / 4), c4 = e % (kKC / 4);
            const long q = q0 + 4 * c4;
            const int t = t0 + row;
            const bool ok = (t < T) && (q < K);
            cp_async16(xs + row * kKC + 4 * c4, ok ? x + (size_t)t * K + q : x, ok ? 16 : 0);
        }
        for (int e = threadIdx.x; e < G::R * (kKC / 4); e += G::NT) {
            const int row = e / (kKC / 4), c4 = e % (kKC / 4);
            const long q = q0 + 4 * c4;
            const bool ok = q < K;
            cp_async16(ws + row * kKC + 4 * c4, ok ? fn_w + (size_t)row * K + q : fn_w, ok ? 16 : 0);
        }
        cp_async_commit();
    };

    float acc[8][S];
    float ss[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ss[i] = 0.f;
#pragma unroll
        for (int r = 0; r < S; ++r)
            acc[i][r] = 0.f;
    }

    if (ck0 < ck1)
        load_chunk(ck0, 0);
    for (int ck = ck0; ck < ck1; ++ck) {
        const int stage = (ck - ck0) & 1;
        if (ck + 1 < ck1) {
            load_chunk(ck + 1, stage ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *xs = sm + stage * G::STAGE;
        const float *ws = xs + G::XS;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const int c = 4 * (kg + 16 * g);
            float4 w[S];
#pragma unroll
            for (int r = 0; r < S; ++r)
                w[r] = *reinterpret_cast<const float4 *>(ws + (r0 + r) * kKC + c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 xv = *reinterpret_cast<const float4 *>(xs + (tg * 8 + i) * kKC + c);
#pragma unroll
                for (int r = 0; r < S; ++r) {
                    acc[i][r] = fmaf(xv.x, w[r].x, acc[i][r]);
                    acc[i][r] = fmaf(xv.y, w[r].y, acc[i][r]);
                    acc[i][r] = fmaf(xv.z, w[r].z, acc[i][r]);
                    acc[i][r] = fmaf(xv.w, w[r].w, acc[i][r]);
                }
                if (warp == 0) {
                    ss[i] = fmaf(xv.x, xv.x, ss[i]);
                    ss[i] = fmaf(xv.y, xv.y, ss[i]);
                    ss[i] = fmaf(xv.z, xv.z, ss[i]);
                    ss[i] = fmaf(xv.w, xv.w, ss[i]);
                }
            }
        }
        __syncthreads();   // this stage is refilled two chunks from now
    }

    // Sum the 16 K-groups of each half-warp: xor butterfly, same tree for every value.
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int r = 0; r < S; ++r)
                acc[i][r] += __shfl_xor_sync(0xffffffffu, acc[i][r], m);
            if (warp == 0)
                ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], m);
        }
    }
    if (kg == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = t0 + tg * 8 + i;
            if (t < T) {
                float *p = part + ((size_t)ks * T + t) * (G::R + 1);
#pragma unroll
                for (int r = 0; r < S; ++r)
                    p[r0 + r] = acc[i][r];
                if (warp == 0)
                    p[G::R] = ss[i];
            }
        }
    }
}

// Sinkhorn of one token (warp 0 of its block): lane j < S holds row j of
// exp(comb logits); every round divides rows, then columns, by (sum + eps).
template <int S>
__device__ __forceinline__ void sinkhorn_comb(const float *mix, float rinv, const float *__restrict__ scale,
                                              const float *__restrict__ base, int iters, float eps, int lane,
                                              float *cm, float *cinv, float *__restrict__ comb_t)
{
    float c[S];
    if (lane < S) {
#pragma unroll
        for (int k = 0; k < S; ++k) {
            const int r = 2 * S + lane * S + k;
            c[k] = expf(mix[r] * rinv * scale[2] + base[r]);
        }
    }
    for (int it = 0; it < iters; ++it) {
        if (lane < S) {
            float rs = 0.f;
#pragma unroll
            for (int k = 0; k < S; ++k)
                rs += c[k];
            const float inv = 1.f / (rs + eps);
#pragma unroll
            for (int k = 0; k < S; ++k) {
                c[k] *= inv;
                cm[lane * S + k] = c[k];
            }
        }
        __syncwarp();
        if (lane < S) {
            float cs = 0.f;
#pragma unroll
            for (int j = 0; j < S; ++j)
                cs += cm[j * S + lane];
            cinv[lane] = 1.f / (cs + eps);
        }
        __syncwarp();
        if (lane < S) {
#pragma unroll
            for (int k = 0; k < S; ++k)
                c[k] *= cinv[k];
        }
        __syncwarp();
    }
    if (lane < S) {
#pragma unroll
        for (int k = 0; k < S; ++k)
            comb_t[lane * S + k] = c[k];
    }
}

// Collapse of one token by its whole block: y[t, :] = sum_c pre_c * x[t, c, :].
template <int S>
__device__ __forceinline__ void collapse_token(const float *__restrict__ x, const float *pre_s, int t, int d,
                                               float *__restrict__ y)
{
    const int d4 = d / 4;
    const float4 *xt = reinterpret_cast<const float4 *>(x + (size_t)t * S * d);
    float4 *yt = reinterpret_cast<float4 *>(y + (size_t)t * d);
    for (int i = threadIdx.x; i < d4; i += kFinishThreads) {
        float4 v = xt[i];
        float4 a = make_float4(pre_s[0] * v.x, pre_s[0] * v.y, pre_s[0] * v.z, pre_s[0] * v.w);
#pragma unroll
        for (int c2 = 1; c2 < S; ++c2) {
            v = xt[(size_t)c2 * d4 + i];
            a.x = fmaf(pre_s[c2], v.x, a.x);
            a.y = fmaf(pre_s[c2], v.y, a.y);
            a.z = fmaf(pre_s[c2], v.z, a.z);
            a.w = fmaf(pre_s[c2], v.w, a.w);
        }
        yt[i] = a;
    }
}

// One block per token: reduce the K slices, gates, Sinkhorn (sites), collapse.
template <int S, bool HEAD>
__global__ void __launch_bounds__(kFinishThreads)
finish_collapse_kernel(const float *__restrict__ part, int nks, const float *__restrict__ x,
                       const float *__restrict__ scale, const float *__restrict__ base, int T,
                       int d, int iters, float eps, float *__restrict__ pre_out,
                       float *__restrict__ post_out, float *__restrict__ comb_out,
                       float *__restrict__ y)
{
    constexpr int R = Geo<S, HEAD>::R;
    __shared__ float mix[R + 1];
    __shared__ float pre_s[S];
    __shared__ float cm[S * S];
    __shared__ float cinv[S];
    const int t = blockIdx.x;
    const int tid = threadIdx.x;

    if (tid < R + 1) {
        float a = 0.f;
        for (int k = 0; k < nks; ++k)
            a += part[((size_t)k * T + t) * (R + 1) + tid];
        mix[tid] = a;
    }
    __syncthreads();

    if (tid < 32) {
        const int lane = tid;
        // rsqrt(mean(x^2) + eps) over the whole s*d slab (rowsq_scale).
        const float rinv = rsqrtf(mix[R] / (float)(S * d) + eps);
        if (lane < (HEAD ? S : 2 * S)) {
            const float l = mix[lane] * rinv * scale[lane < S ? 0 : 1] + base[lane];
            const float sg = 1.f / (1.f + expf(-l));
            if (lane < S) {
                const float p = sg + eps;
                if (pre_out)   // the head's gates are an optional output
                    pre_out[(size_t)t * S + lane] = p;
                pre_s[lane] = p;
            } else {
                post_out[(size_t)t * S + (lane - S)] = 2.f * sg;
            }
        }
        if (!HEAD)
            sinkhorn_comb<S>(mix, rinv, scale, base, iters, eps, lane, cm, cinv, comb_out + (size_t)t * S * S);
    }
    __syncthreads();
    collapse_token<S>(x, pre_s, t, d, y);
}

template <int S, bool HEAD>
cudaError_t run_generic(const float *x, const float *fn_w, const float *scale, const float *base,
                        int T, int d, int iters, float eps, float *pre, float *post, float *comb,
                        float *y, void *workspace, cudaStream_t st)
{
    using G = Geo<S, HEAD>;
    const Split sp = make_split(T, S, d);
    float *part = reinterpret_cast<float *>(static_cast<char *>(workspace) + kStatusBytes);
    if (G::SMEM > 48 * 1024) {
        // The dynamic shared-memory limit is a per-context attribute: set once per
        // device and context (a device reset replaces the context and drops it).
        static std::mutex mu;
        static unsigned long long set_in[64] = {};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
            return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long ctx = context_id();
        if (ctx == 0 || set_in[dev] != ctx) {
            cudaError_t e = cudaFuncSetAttribute(mixes_partial_kernel<S, HEAD>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G::SMEM);
            if (e != cudaSuccess)
                return e;
            set_in[dev] = context_id();
        }
    }
    dim3 grid1(sp.nt, sp.nks);
    mixes_partial_kernel<S, HEAD><<<grid1, G::NT, G::SMEM, st>>>(x, fn_w, T, S * d, sp.nck, sp.ck_per, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    finish_collapse_kernel<S, HEAD><<<T, kFinishThreads, 0, st>>>(part, sp.nks, x, scale, base, T, d, iters,
                                                            eps, pre, post, comb, y);
    return cudaGetLastError();
}

}  // namespace

size_t generic_workspace_bytes(int T, int s, int d)
{
    const Split sp = make_split(T, s, d);
    const int R = (2 + s) * s;
    return kStatusBytes + (size_t)sp.nks * (size_t)T * (size_t)(R + 1) * sizeof(float);
}

cudaError_t launch_pre_generic(const float *x, const float *fn_w, const float *scale,
                               const float *base, int T, int s, int d, int iters, float eps,
                               float *pre, float *post, float *comb, float *y, void *workspace,
                               cudaStream_t st)
{
    switch (s) {
#define HC_CASE(S)                                                                              \
    case S:                                                                                     \
        return run_generic<S, false>(x, fn_w, scale, base, T, d, iters, eps, pre, post, comb, y, \
                                     workspace, st);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4) HC_CASE(5) HC_CASE(6) HC_CASE(7) HC_CASE(8)
#undef HC_CASE
    default:
        return cudaErrorInvalidValue;
    }
}

cudaError_t launch_head_generic(const float *x, const float *fn_w, const float *scale,
                                const float *base, int T, int s, int d, float eps, float *gates,
                                float *y, void *workspace, cudaStream_t st)
{
    switch (s) {
#define HC_CASE(S)                                                                               \
    case S:                                                                                      \
        return run_generic<S, true>(x, fn_w, scale, base, T, d, 1, eps, gates, nullptr, nullptr, y, \
                                    workspace, st);
        HC_CASE(1) HC_CASE(2) HC_CASE(3) HC_CASE(4) HC_CASE(5) HC_CASE(6) HC_CASE(7) HC_CASE(8)
#undef HC_CASE
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace hc
