// hc_stream_ops.cu -- the HBM-streaming kernels of the site program:
//   hc_post   x'[t,k,:] = post[t,k] * f[t,:] + sum_j comb[t,j,k] * x[t,j,:]
//             (memra-engine hyper.rs page, `post`; module header last line)
//   hc_expand x[t,c,:]  = emb[t,:]            (hyper.rs `expand`)
//   hc_mean   out[t,:]  = mean_c x[t,c,:]     (hyper.rs `contract_mean`)
//
// Each is bound by HBM bandwidth (hc_post: ~1.1 FLOP per byte), so the design
// is about bytes in flight: one thread owns one 16-byte column group of one
// token and touches every stream of it, so each x element is read exactly once
// and each output element written once, with 128-bit coalesced accesses.  A
// block covers kColsPerBlock float4 groups of a single token, which lets the
// token's post/comb coefficients sit in shared memory (one load per block,
// broadcast reads after that) instead of s + s*s loads per thread.
#include "hc_internal.cuh"

namespace hc {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float4 ld_stream(const float4 *p)
{
    // Read-once data: keep it out of L1 and mark it evict-first in L2.
    return __ldcs(p);
}

template <int S>
__global__ void __launch_bounds__(kThreads)
hc_post_kernel(const float4 *__restrict__ x, const float4 *__restrict__ f,
               const float *__restrict__ post, const float *__restrict__ comb,
               float4 *__restrict__ x_out, int d4, int blocks_per_token)
{
    __shared__ float coef[S + S * S];   // post[k] then comb[j][k]
    const int t = blockIdx.x / blocks_per_token;
    const int col = (blockIdx.x - t * blocks_per_token) * kThreads + threadIdx.x;
    // Up to six streams the streaming loads go out before the coefficient barrier, so
    // their latency covers the coefficients'; with more, holding them across it would
    // cost a resident block per SM (registers), and they follow it.
    constexpr bool kEarly = S <= 6;
    const bool active = col < d4;
    const size_t xbase = (size_t)t * S * d4 + col;
    float4 xv[S], fv = make_float4(0.f, 0.f, 0.f, 0.f);
    auto load = [&]() {
#pragma unroll
        for (int j = 0; j < S; ++j)
            xv[j] = ld_stream(x + xbase + (size_t)j * d4);
        fv = ld_stream(f + (size_t)t * d4 + col);
    };
    if (kEarly && active)
        load();
    if (threadIdx.x < S)
        coef[threadIdx.x] = post[(size_t)t * S + threadIdx.x];
    else if (threadIdx.x < S + S * S)
        coef[threadIdx.x] = comb[(size_t)t * S * S + (threadIdx.x - S)];
    __syncthreads();
    if (!active)
        return;
    if (!kEarly)
        load();

#pragma unroll
    for (int k = 0; k < S; ++k) {
        const float pk = coef[k];
        float4 o = make_float4(pk * fv.x, pk * fv.y, pk * fv.z, pk * fv.w);
#pragma unroll
        for (int j = 0; j < S; ++j) {
            const float c = coef[S + j * S + k];
            o.x = fmaf(c, xv[j].x, o.x);
            o.y = fmaf(c, xv[j].y, o.y);
            o.z = fmaf(c, xv[j].z, o.z);
            o.w = fmaf(c, xv[j].w, o.w);
        }
        x_out[xbase + (size_t)k * d4] = o;
    }
}

template <int S>
__global__ void __launch_bounds__(kThreads)
hc_expand_kernel(const float4 *__restrict__ emb, float4 *__restrict__ x, int d4, size_t n4)
{
    const size_t g = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (g >= n4)
        return;
    const size_t t = g / d4, col = g - t * d4;
    const float4 v = ld_stream(emb + g);
#pragma unroll
    for (int c = 0; c < S; ++c)
        x[(t * S + c) * d4 + col] = v;
}

template <int S>
__global__ void __launch_bounds__(kThreads)
hc_mean_kernel(const float4 *__restrict__ x, float4 *__restrict__ out, int d4, size_t n4)
{
    const size_t g = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (g >= n4)
        return;
    const size_t t = g / d4, col = g - t * d4;
    float4 a = ld_stream(x + (t * S) * d4 + col);
#pragma unroll
    for (int c = 1; c < S; ++c) {
        const float4 v = ld_stream(x + (t * S + c) * d4 + col);
        a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
    }
    const float inv_s = (float)S;
    out[g] = make_float4(a.x / inv_s, a.y / inv_s, a.z / inv_s, a.w / inv_s);
}

template <template <int> class Launcher, typename... Args>
cudaError_t by_streams(int s, Args... args)
{
    switch (s) {
    case 1: return Launcher<1>::run(args...);
    case 2: return Launcher<2>::run(args...);
    case 3: return Launcher<3>::run(args...);
    case 4: return Launcher<4>::run(args...);
    case 5: return Launcher<5>::run(args...);
    case 6: return Launcher<6>::run(args...);
    case 7: return Launcher<7>::run(args...);
    case 8: return Launcher<8>::run(args...);
    default: return cudaErrorInvalidValue;
    }
}

template <int S>
struct PostLaunch {
    static cudaError_t run(const float *x, const float *f, const float *post, const float *comb,
                           float *x_out, int T, int d, cudaStream_t st)
    {
        const int d4 = d / 4;
        const int bpt = (d4 + kThreads - 1) / kThreads;
        hc_post_kernel<S><<<(unsigned)((size_t)T * bpt), kThreads, 0, st>>>(
            reinterpret_cast<const float4 *>(x), reinterpret_cast<const float4 *>(f), post, comb,
            reinterpret_cast<float4 *>(x_out), d4, bpt);
        return cudaGetLastError();
    }
};

template <int S>
struct ExpandLaunch {
    static cudaError_t run(const float *emb, float *x, int T, int d, cudaStream_t st)
    {
        const size_t n4 = (size_t)T * (d / 4);
        hc_expand_kernel<S><<<(unsigned)((n4 + kThreads - 1) / kThreads), kThreads, 0, st>>>(
            reinterpret_cast<const float4 *>(emb), reinterpret_cast<float4 *>(x), d / 4, n4);
        return cudaGetLastError();
    }
};

template <int S>
struct MeanLaunch {
    static cudaError_t run(const float *x, float *out, int T, int d, cudaStream_t st)
    {
        const size_t n4 = (size_t)T * (d / 4);
        hc_mean_kernel<S><<<(unsigned)((n4 + kThreads - 1) / kThreads), kThreads, 0, st>>>(
            reinterpret_cast<const float4 *>(x), reinterpret_cast<float4 *>(out), d / 4, n4);
        return cudaGetLastError();
    }
};

}  // namespace

cudaError_t launch_post(const float *x, const float *f, const float *post, const float *comb,
                        float *x_out, int T, int s, int d, cudaStream_t st)
{
    return by_streams<PostLaunch>(s, x, f, post, comb, x_out, T, d, st);
}

cudaError_t launch_expand(const float *emb, float *x, int T, int s, int d, cudaStream_t st)
{
    return by_streams<ExpandLaunch>(s, emb, x, T, d, st);
}

cudaError_t launch_mean(const float *x, float *out, int T, int s, int d, cudaStream_t st)
{
    return by_streams<MeanLaunch>(s, x, out, T, d, st);
}

}  // namespace hc
