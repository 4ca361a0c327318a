// hc_norm.cu -- the branch-input norm of the collapse and its int8 pair.
//
// What it computes (memra-engine hyper.rs page, module header: f = branch(rms_norm(y));
// the pages' fused v4z pre kernel emits the norm with an int8 pair for the branch):
//   z[t, i] = y[t, i] * rsqrt(mean_i(y[t, :]^2) + eps_norm) * norm_w[i]
//   optionally, per block of 32 consecutive z of a token (GGML's Q8_0 layout):
//     scale = amax / 127,  q = round-half-away(z * (1 / scale)), 0 when scale is 0.
// One block of 256 threads per token; thread i holds float4 columns i, i+256, ...
// The sum of squares has a fixed order (per-thread in column order, then an xor
// tree over the warp, then the 8 warps in order), so results are bit-identical run
// to run.  The int8 codes are decided with IEEE float32 division, reciprocal and
// multiply (no contraction), the same operations as the float32 quantiser they are
// checked against.
#include "hc_internal.cuh"

namespace hc {
namespace {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
rms_norm_q8_kernel(const float4 *__restrict__ y, const float4 *__restrict__ norm_w, int d4, float eps_norm,
                   float inv_d, float4 *__restrict__ z, char4 *__restrict__ q, float *__restrict__ q_scale)
{
    __shared__ float warp_ss[kNormThreads / 32];
    const int t = blockIdx.x;
    const float4 *yt = y + (size_t)t * d4;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d4; i += kNormThreads) {
        const float4 v = yt[i];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
        ss += __shfl_xor_sync(0xffffffffu, ss, m);
    if ((threadIdx.x & 31) == 0)
        warp_ss[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w)
        tot += warp_ss[w];
    const float r = rsqrtf(tot * inv_d + eps_norm);

    for (int i0 = 0; i0 < d4; i0 += kNormThreads) {
        const int i = i0 + threadIdx.x;
        float4 zv = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < d4) {
            const float4 v = yt[i];
            const float4 w = norm_w[i];
            zv = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
            z[(size_t)t * d4 + i] = zv;
        }
        if (q) {
            // 8 consecutive threads hold one block of 32 (d % 32 == 0, so a block
            // never straddles the row end, and i0 is a multiple of 8).
            float amax = fmaxf(fmaxf(fabsf(zv.x), fabsf(zv.y)), fmaxf(fabsf(zv.z), fabsf(zv.w)));
#pragma unroll
            for (int m = 1; m < 8; m <<= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
            if (i < d4) {
                const float sc = __fdiv_rn(amax, 127.0f);
                const float inv = sc != 0.0f ? __frcp_rn(sc) : 0.0f;
                auto code = [&](float a) {
                    const float rv = fminf(fmaxf(roundf(__fmul_rn(a, inv)), -127.0f), 127.0f);
                    return (signed char)rv;
                };
                q[(size_t)t * d4 + i] = make_char4(code(zv.x), code(zv.y), code(zv.z), code(zv.w));
                if ((i & 7) == 0)
                    q_scale[(size_t)t * (d4 / 8) + (i >> 3)] = sc;
            }
        }
    }
}

}  // namespace

cudaError_t launch_rms_norm_q8(const float *y, const float *norm_w, int T, int d, float eps_norm, float *z,
                               signed char *q, float *q_scale, cudaStream_t st)
{
    const int d4 = d / 4;
    rms_norm_q8_kernel<<<T, kNormThreads, 0, st>>>(
        reinterpret_cast<const float4 *>(y), reinterpret_cast<const float4 *>(norm_w), d4, eps_norm,
        1.0f / (float)d, reinterpret_cast<float4 *>(z), reinterpret_cast<char4 *>(q), q_scale);
    return cudaGetLastError();
}

}  // namespace hc
