/*
 * hc_oracle.c -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * A plain, slow, float64 CPU restatement of the mHC (manifold-constrained
 * hyper-connections) site program.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg load this library; the CUDA library never
 * links, includes or calls it, and this file includes nothing of the CUDA
 * library.  Inputs arrive as float64 (callers widen float32 bytes), every
 * intermediate is float64, and each step follows the formulas of the
 * memra-engine "hyper.rs" page (module header, "ARITHMETIC CONTRACT"):
 *
 *   mixes[t, :]   = fn_w . x[t, :, :]                  rows = (2+s)*s
 *   mixes[t, :]  *= rsqrt(mean(x[t]^2) + eps)          over the whole s*d slab
 *   pre/post/comb = sinkhorn(mixes[t, :], scale, base)
 *   y[t, :]       = sum_c pre[t, c] * x[t, c, :]
 *   x'[t, k, :]   = post[t, k] * f[t, :] + sum_j comb[t, j, k] * x[t, j, :]
 *
 * The pages never print the split itself.  The reading used (and pinned by
 * the tests against closed forms) is:
 *   logit[r] = mixes[r] * scale[group(r)] + base[r], group 0 = pre rows
 *              (r < s), 1 = post rows (s <= r < 2s), 2 = comb rows
 *              ("three gate scales -- pre, post, combination", hyper.rs
 *              load_site; row order pre, post, comb from HyperTopology::rows);
 *   pre[c]   = sigmoid(logit[c]) + eps;  post[c] = 2 * sigmoid(logit[s+c]);
 *   C[j][k]  = exp(logit[2s + j*s + k]); then `iters` times: divide every row
 *              by (row sum + eps), then every column by (column sum + eps);
 *              comb[j][k] = C[j][k].  No max-subtraction in exp.
 * The same eps (the topology's hc eps) is used in the rsqrt, in pre and in
 * both Sinkhorn denominators (hyper.rs pre_finish_into passes one eps to
 * rowsq_scale and to hc_sinkhorn_m).
 *
 * The gated-head trunk exit (hco_head) is the pre gate and collapse of a head
 * whose rows equal its streams, with one scale; see its comment.
 *
 * Parity status: every exported function is pinned by tests/test_oracle_pins.py
 * (closed forms, hand-derived golden values, invariants, brute force).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define HCO_OK 0
#define HCO_EINVAL 1
#define HCO_ENOMEM 2

int hco_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* Row r of the mixes block belongs to scale group 0 (pre), 1 (post) or 2 (comb). */
static int row_group(long r, int s) { return r < s ? 0 : (r < 2 * s ? 1 : 2); }

/*
 * One token of the pre-chain (hyper.rs module header, lines "mixes ...",
 * "mixes *= rsqrt ...", "pre/post/comb = sinkhorn ...", "y = ...").
 * xt: [s, d] slab; fn_w: [R, s*d] row-major; work: >= R + s*s doubles.
 */
static void pre_token(const double *xt, const double *fn_w, const double *scale,
                      const double *base, int s, long d, int iters, double eps,
                      double *pre, double *post, double *comb, double *y,
                      double *mixes_out, double *logits_out, double *work)
{
    const long K = (long)s * d;
    const long R = (long)(2 + s) * s;
    double *logit = work;          /* [R]   */
    double *C = work + R;          /* [s*s] */

    /* 1. mean of squares over the whole s*d slab, then rsqrt(mean + eps). */
    double ss = 0.0;
    for (long q = 0; q < K; ++q)
        ss += xt[q] * xt[q];
    const double rinv = 1.0 / sqrt(ss / (double)K + eps);

    /* 2. mixes[r] = rinv * (fn_w[r, :] . x[t]) ; 3. logits. */
    for (long r = 0; r < R; ++r) {
        const double *wr = fn_w + r * K;
        double dot = 0.0;
        for (long q = 0; q < K; ++q)
            dot += wr[q] * xt[q];
        const double m = rinv * dot;
        if (mixes_out)
            mixes_out[r] = m;
        logit[r] = m * scale[row_group(r, s)] + base[r];
        if (logits_out)
            logits_out[r] = logit[r];
    }

    /* 4. gates. */
    for (int c = 0; c < s; ++c) {
        pre[c] = sigmoid(logit[c]) + eps;
        post[c] = 2.0 * sigmoid(logit[s + c]);
    }

    /* 5. Sinkhorn: exp, then `iters` x (rows, then columns), eps in each denominator. */
    for (int j = 0; j < s; ++j)
        for (int k = 0; k < s; ++k)
            C[j * s + k] = exp(logit[2 * s + j * s + k]);
    for (int it = 0; it < iters; ++it) {
        for (int j = 0; j < s; ++j) {
            double rs = 0.0;
            for (int k = 0; k < s; ++k)
                rs += C[j * s + k];
            for (int k = 0; k < s; ++k)
                C[j * s + k] /= (rs + eps);
        }
        for (int k = 0; k < s; ++k) {
            double cs = 0.0;
            for (int j = 0; j < s; ++j)
                cs += C[j * s + k];
            for (int j = 0; j < s; ++j)
                C[j * s + k] /= (cs + eps);
        }
    }
    memcpy(comb, C, sizeof(double) * (size_t)s * (size_t)s);

    /* 6. collapse: y[i] = sum_c pre[c] * x[c, i]. */
    for (long i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int c = 0; c < s; ++c)
            acc += pre[c] * xt[(long)c * d + i];
        y[i] = acc;
    }
}

/*
 * The pre-chain over T tokens.  x [T, s, d], fn_w [R, s*d], scale [3],
 * base [R] -> pre [T, s], post [T, s], comb [T, s, s], y [T, d];
 * mixes / logits [T, R] are optional (NULL to skip).
 */
int hco_pre(const double *x, const double *fn_w, const double *scale, const double *base,
            long T, int s, long d, int iters, double eps,
            double *pre, double *post, double *comb, double *y,
            double *mixes, double *logits, int nthreads)
{
    if (T < 0 || s < 1 || d < 1 || iters < 0 || !(eps >= 0.0))
        return HCO_EINVAL;
    if (T == 0)
        return HCO_OK;
    if (!x || !fn_w || !scale || !base || !pre || !post || !comb || !y)
        return HCO_EINVAL;
    const long R = (long)(2 + s) * s;
    int failed = 0;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *work = (double *)malloc(sizeof(double) * (size_t)(R + (long)s * s));
        if (!work) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (long t = 0; t < T; ++t)
                pre_token(x + t * s * d, fn_w, scale, base, s, d, iters, eps,
                          pre + t * s, post + t * s, comb + t * s * s, y + t * d,
                          mixes ? mixes + t * R : NULL, logits ? logits + t * R : NULL, work);
            free(work);
        }
    }
    return failed ? HCO_ENOMEM : HCO_OK;
}

/*
 * hc_post (hyper.rs `post`): out[t, k, i] = post[t, k] * f[t, i]
 *                                           + sum_j comb[t, j, k] * x[t, j, i].
 * x is the site's INPUT stream state (the residual), not the layer's.
 */
int hco_post(const double *x, const double *f, const double *post, const double *comb,
             double *x_out, long T, int s, long d, int nthreads)
{
    if (T < 0 || s < 1 || d < 1)
        return HCO_EINVAL;
    if (T == 0)
        return HCO_OK;
    if (!x || !f || !post || !comb || !x_out)
        return HCO_EINVAL;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (long t = 0; t < T; ++t) {
        const double *xt = x + t * s * d;
        const double *ct = comb + t * s * s;
        for (int k = 0; k < s; ++k) {
            double *ot = x_out + (t * s + k) * d;
            for (long i = 0; i < d; ++i) {
                double acc = post[t * s + k] * f[t * d + i];
                for (int j = 0; j < s; ++j)
                    acc += ct[j * s + k] * xt[(long)j * d + i];
                ot[i] = acc;
            }
        }
    }
    return HCO_OK;
}

/*
 * Gated-head trunk exit (hyper.rs `collapse`, case HcCollapse::GatedHead; the
 * head trio of HyperHead::load: fn_w [s, s*d] -- rows equal to streams -- base [s]
 * and ONE scale).  The pages chain a linear (mixes = fn_w . x[t]), rowsq_scale
 * (mixes *= rsqrt(mean(x[t]^2) + eps)), hc_head_pre (gates) and hc_collapse
 * (y = sum_c gate_c * x[t, c, :]); they print no formula for the gates.  The
 * reading used is the site's pre gate with the head's single scale:
 *   gate[c] = sigmoid(mixes[c] * scale + base[c]) + eps.
 * x [T, s, d], fn_w [s, s*d], scale [1], base [s] -> gates [T, s], y [T, d].
 */
int hco_head(const double *x, const double *fn_w, const double *scale, const double *base,
             long T, int s, long d, double eps, double *gates, double *y, int nthreads)
{
    if (T < 0 || s < 1 || d < 1 || !(eps >= 0.0))
        return HCO_EINVAL;
    if (T == 0)
        return HCO_OK;
    if (!x || !fn_w || !scale || !base || !gates || !y)
        return HCO_EINVAL;
    if (nthreads < 1)
        nthreads = 1;
    const long K = (long)s * d;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (long t = 0; t < T; ++t) {
        const double *xt = x + t * K;
        double ss = 0.0;
        for (long q = 0; q < K; ++q)
            ss += xt[q] * xt[q];
        const double rinv = 1.0 / sqrt(ss / (double)K + eps);
        double *g = gates + t * s;
        for (int c = 0; c < s; ++c) {
            const double *wr = fn_w + (long)c * K;
            double dot = 0.0;
            for (long q = 0; q < K; ++q)
                dot += wr[q] * xt[q];
            g[c] = sigmoid(rinv * dot * scale[0] + base[c]) + eps;
        }
        for (long i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int c = 0; c < s; ++c)
                acc += g[c] * xt[(long)c * d + i];
            y[t * d + i] = acc;
        }
    }
    return HCO_OK;
}

/*
 * Branch-input norm of the collapse (hyper.rs module header: f = branch(rms_norm(y));
 * the pages' fused v4z variant of the pre kernel also emits it, with an int8 pair):
 *   z[t, i] = y[t, i] * rsqrt(mean_i(y[t, :]^2) + eps_norm) * norm_w[i]     (float64)
 * y [T, d], norm_w [d] -> z [T, d].
 */
int hco_rms_norm(const double *y, const double *norm_w, long T, long d, double eps_norm, double *z)
{
    if (T < 0 || d < 1 || !(eps_norm >= 0.0))
        return HCO_EINVAL;
    for (long t = 0; t < T; ++t) {
        const double *yt = y + t * d;
        double ss = 0.0;
        for (long i = 0; i < d; ++i)
            ss += yt[i] * yt[i];
        const double r = 1.0 / sqrt(ss / (double)d + eps_norm);
        for (long i = 0; i < d; ++i)
            z[t * d + i] = yt[i] * r * norm_w[i];
    }
    return HCO_OK;
}

/*
 * The int8 pair of that norm, read as GGML's Q8_0 blocks of 32 values (the pages
 * allocate an int8 [d] and a float [d/32] for it): per block, amax = max |z|,
 * scale = amax / 127, q = round(z * (1 / scale)) (0 when scale is 0), rounding half
 * away from zero.  These steps decide integers, so they run in float32, on float32
 * z, in exactly this order: a float64 restatement could round a code differently.
 * z [n] float32 (n % 32 == 0) -> q [n] int8, scale [n / 32] float32.
 */
int hco_q8_blocks_f32(const float *z, long n, signed char *q, float *scale)
{
    if (n < 0 || n % 32)
        return HCO_EINVAL;
    for (long b = 0; b < n / 32; ++b) {
        const float *zb = z + b * 32;
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            const float a = fabsf(zb[i]);
            if (a > amax)
                amax = a;
        }
        const float sc = amax / 127.0f;
        const float inv = sc != 0.0f ? 1.0f / sc : 0.0f;
        scale[b] = sc;
        for (int i = 0; i < 32; ++i) {
            const float v = zb[i] * inv;
            float r = roundf(v);
            if (r > 127.0f)
                r = 127.0f;
            if (r < -127.0f)
                r = -127.0f;
            q[b * 32 + i] = (signed char)r;
        }
    }
    return HCO_OK;
}

/* hc_expand (hyper.rs `expand`): every stream starts as the token's embedding. */
int hco_expand(const double *emb, double *x, long T, int s, long d)
{
    if (T < 0 || s < 1 || d < 1)
        return HCO_EINVAL;
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < s; ++c)
            for (long i = 0; i < d; ++i)
                x[(t * s + c) * d + i] = emb[t * d + i];
    return HCO_OK;
}

/* hc_mean (hyper.rs `contract_mean`): unweighted mean over the s streams. */
int hco_mean(const double *x, double *out, long T, int s, long d)
{
    if (T < 0 || s < 1 || d < 1)
        return HCO_EINVAL;
    for (long t = 0; t < T; ++t)
        for (long i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int c = 0; c < s; ++c)
                acc += x[(t * s + c) * d + i];
            out[t * d + i] = acc / (double)s;
        }
    return HCO_OK;
}
