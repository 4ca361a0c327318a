/*
 * hc.h -- C ABI of the GB300 (sm_103a) mHC site-program library.
 *
 * mHC (manifold-constrained hyper-connections) carries a residual stream state
 * x[T, s, d] of s parallel streams per token.  Each site (attention, then MLP,
 * of every layer) runs, per token, the program given in the module header of
 * the memra-engine "hyper.rs" page ("ARITHMETIC CONTRACT"):
 *
 *   mixes[t, :]   = fn_w . x[t, :, :]                  rows R = (2+s)*s
 *   mixes[t, :]  *= rsqrt(mean(x[t]^2) + eps)          over the whole s*d slab
 *   pre/post/comb = sinkhorn(mixes[t, :], scale, base)
 *   y[t, :]       = sum_c pre[t, c] * x[t, c, :]
 *   f             = branch(rms_norm(y))                (not part of this library)
 *   x'[t, k, :]   = post[t, k] * f[t, :] + sum_j comb[t, j, k] * x[t, j, :]
 *
 * The split, which the pages never print, is read as:
 *   logit[r] = mixes[r] * scale[g(r)] + base[r], g = 0 for the s pre rows,
 *              1 for the s post rows, 2 for the s*s comb rows (that row order);
 *   pre  = sigmoid(logit) + eps,  post = 2 * sigmoid(logit),
 *   comb = exp(logit[2s + j*s + k]) then `iters` rounds of (divide each row by
 *          its sum + eps; divide each column by its sum + eps).
 *
 * Conventions (all entry points):
 *   - Layout is token-major: element (t, k, i) of a [T, s, d] state is at
 *     (t*s + k)*d + i, so one token's s*d slab is contiguous (hyper.rs module
 *     header, "MEMORY LAYOUT").  fn_w is row-major [R, s*d].
 *   - Every tensor pointer is a DEVICE pointer to float32 owned by the caller.
 *     The library never allocates, never frees and never synchronises; all
 *     work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Outputs are fully overwritten; inputs are never written.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-zero return means nothing was enqueued, except HC_ERR_CUDA, which
 *     reports the error of the launch itself.
 *   - T == 0 is a valid empty batch: nothing is launched and HC_OK returned.
 *   - Limits: 1 <= s <= 8 (the pages' fused kernels size their shared arrays
 *     for hc <= 8), d >= 4 and d % 4 == 0, iters >= 1, eps > 0 and finite
 *     (HyperTopology::from_plan refuses streams == 0, epsilon <= 0 and zero
 *     iterations), T*s*d < 2^31.
 *   - Pointers to x, fn_w, y, f, x_out, emb and out must be 16-byte aligned
 *     (vector and bulk-copy access); pre, post, comb, scale and base 4-byte.
 */
#ifndef MHC_GB300_HC_H
#define MHC_GB300_HC_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum hc_status {
    HC_OK = 0,
    HC_ERR_NULL = 1,        /* a required pointer is NULL                            */
    HC_ERR_DIM = 2,         /* T, s, d, iters or eps outside the limits above        */
    HC_ERR_ALIGN = 3,       /* pointer misaligned, or d % 4 != 0                     */
    HC_ERR_ALIAS = 4,       /* an output overlaps an input or another output         */
    HC_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than hc_pre_workspace_bytes */
    HC_ERR_CUDA = 6,        /* the CUDA runtime reported an error                    */
    HC_ERR_DEVICE = 7,      /* a kernel flagged an error in the workspace status word */
    HC_ERR_UNSUPPORTED = 8, /* the requested kernel path cannot run this shape here  */
    HC_ERR_TOO_LARGE = 9    /* hc_pre_fused_noalloc: shape needs more scratch than its
                               static buffer holds                                   */
};

/* Kernel paths of hc_pre_fused_path. */
enum hc_pre_path {
    HC_PATH_AUTO = 0,     /* what hc_pre_fused runs                                   */
    HC_PATH_GENERIC = 1,  /* any supported shape: split-K mixes kernel + finish kernel */
    HC_PATH_CLUSTER = 2,  /* one fused launch, x read once: thread-block clusters split
                             the hidden dimension (at prefill sizes with the helper
                             kernel beside it: hc_pre_helper_tokens); needs s <= 4 and
                             s*d <= 16384 with d % 64 == 0                             */
    HC_PATH_WIDE = 3      /* one fused launch over every SM, x read once from HBM, for
                             5 <= s <= 8: each CTA keeps a fixed hidden range of fn_w
                             resident.  Needs d split over at least 32 CTAs (at most one
                             per SM) into widths that are multiples of the unit u (the
                             smallest multiple of 8 with s*u % 64 == 0: 64, 32, 64, 8 for
                             s = 5..8), at most one unit apart and balanced to 3/4, with
                             the slice fitting TMEM and shared memory (e.g. s = 8 with
                             d = 7168 or 4096, s = 5..7 with d = 4096, s = 5 or 7 with
                             d = 7168; not s = 6 with d = 7168);
                             hc_pre_auto_path says whether it runs a shape             */
};

/* Human-readable name of a status code (static string, never NULL). */
const char *hc_status_string(int rc);

/*
 * hc_expand -- model entry: [T, d] embeddings -> [T, s, d] stream state, every
 * stream a copy of the token's embedding (hyper.rs `expand`; the pages give
 * only the shapes, replication is the reading used).
 *   emb [T, d] (in), x [T, s, d] (out, must not overlap emb).
 */
int hc_expand(const float *emb, float *x, int T, int s, int d, void *stream);

/*
 * Bytes of device workspace hc_pre_fused needs for this shape (the most any
 * path needs; each call checks ws_bytes against the path it runs).  The
 * workspace holds a status word (first 256 bytes) and, by path: on the generic
 * path split-K partial sums; on the wide path the tiles' counters and flags
 * (zeroed by the call itself, on its stream, before its launch) and per-CTA
 * partial slots; on the cluster path at prefill sizes the helper kernel's
 * partial sums (a smaller workspace, down to the 256-byte status word, only
 * keeps the helper from running: see hc_pre_helper_tokens).  It must be zeroed
 * once before first use (hc_workspace_init);
 * every call leaves it valid for the next.  Calls that share a workspace must
 * not run concurrently.
 */
size_t hc_pre_workspace_bytes(int T, int s, int d);

/* Zero `ws_bytes` of workspace on `stream` (a cudaMemsetAsync). */
int hc_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/*
 * Read the workspace status word (synchronises `stream`): HC_OK, or
 * HC_ERR_DEVICE if a kernel gave up on a bounded wait.  The word is sticky
 * until hc_workspace_init clears it.  Its first 32-bit field is the code (1: a
 * bounded wait gave up; 2, only in the bounds-checked build of the library: a
 * store outside its buffer was refused), the second the site, the third the
 * reporting block.
 *
 * Outputs are valid only while the word reads HC_OK.  While it is non-zero,
 * every later hc_pre_fused, hc_post_pre_fused and hc_head call on that
 * workspace that runs the cluster or wide path still returns HC_OK (the
 * host cannot see the word without synchronising) but its kernel does
 * nothing: pre, post, comb, y, gates and x_new are left as they were.  The
 * generic path has no waits, never sets the word and runs regardless.
 */
int hc_workspace_status(const void *workspace, void *stream);

/*
 * hc_pre_fused -- the pre-chain of one site (hyper.rs `pre` + `pre_finish_into`,
 * module header lines "mixes", "mixes *= rsqrt", "pre/post/comb = sinkhorn",
 * "y = sum_c pre . x").  Unlike the pages' fused kernels, which take the mixes
 * precomputed by a separate GEMM, this call computes the mixes contraction
 * itself, so each token's slab is read from memory inside the same program.
 *
 *   x     [T, s, d]  stream state (in)
 *   fn_w  [R, s*d]   row-major mixing weights, R = (2+s)*s (in)
 *   scale [3]        gate scales: pre, post, comb (in)
 *   base  [R]        per-row bias (in)
 *   pre   [T, s]     sigmoid gates + eps (out)
 *   post  [T, s]     2 * sigmoid gates (out)
 *   comb  [T, s, s]  Sinkhorn-normalised combination, comb[t, j, k] (out)
 *   y     [T, d]     collapsed branch input (out)
 *   workspace, ws_bytes: device scratch of >= hc_pre_workspace_bytes(T, s, d).
 *   Outputs must not overlap x, fn_w, scale, base or each other.
 * Results are float32 and repeated calls are bit-identical (every sum has a
 * fixed order; no floating-point atomics).  On the cluster and wide paths a
 * token's results are also the same bits whatever else is in the batch; the
 * generic path sizes its K split by T, so there they may differ in the last
 * bits.  Outputs are valid only while hc_workspace_status reads HC_OK (see
 * there: a non-zero status word makes the cluster and wide kernels skip).
 */
int hc_pre_fused(const float *x, const float *fn_w, const float *scale, const float *base,
                 int T, int s, int d, int iters, float eps,
                 float *pre, float *post, float *comb, float *y,
                 void *workspace, size_t ws_bytes, void *stream);

/*
 * hc_pre_fused with an explicit kernel path (enum hc_pre_path).  Returns
 * HC_ERR_UNSUPPORTED if that path cannot run the shape on this device.
 */
int hc_pre_fused_path(const float *x, const float *fn_w, const float *scale, const float *base,
                      int T, int s, int d, int iters, float eps,
                      float *pre, float *post, float *comb, float *y,
                      void *workspace, size_t ws_bytes, void *stream, int path);

/* The path HC_PATH_AUTO picks for this shape on the current device. */
int hc_pre_auto_path(int T, int s, int d);

/*
 * hc_pre_helper_tokens -- on the cluster path at prefill sizes the cluster kernel,
 * whose 16-CTA clusters cannot be placed on every SM, is followed on the stream by a
 * helper kernel on the SMs it leaves free (programmatic dependent launch: both run
 * at once).  The helper takes the batch's last tokens and plays each cluster's 16
 * CTAs in turn with the same arithmetic in the same order, so every token's outputs
 * are the same bits whichever kernel computed them.  This returns how many tokens
 * it takes for a call of this shape on the current device with a workspace of
 * ws_bytes: fused != 0 for hc_post_pre_fused, 0 for hc_pre_fused (the gated head and
 * hc_pre_fused_norm's one-launch mode never use it).  0 means the cluster kernel
 * alone (small T, another path, or a workspace without room for the helper's
 * partials); -1 for dimensions out of range.
 */
int hc_pre_helper_tokens(int T, int s, int d, int fused, size_t ws_bytes);

/*
 * hc_pre_fused_noalloc -- hc_pre_fused for callers that cannot allocate device
 * memory when they run a site: an engine whose device memory is all carved into
 * a fixed arena at start-up, a plugin whose host framework owns every
 * allocation, a latency-critical loop that cannot pay for cudaMalloc/cudaFree
 * (they may block or synchronise the device).  It takes no workspace.  (The
 * pages have no counterpart; this entry point exists for such callers.)
 *
 * Same arguments, layouts, validation and results as hc_pre_fused run on the
 * generic path (HC_PATH_GENERIC), minus workspace and ws_bytes.  The split-K
 * scratch lives in a 4 MiB static device buffer inside the library, which every
 * GPU that loads the library holds until the process exits; shapes whose
 * generic-path scratch (the 256-byte status block and the split-K partial
 * sums) needs more than that (e.g. T above about 41,000 at s = 4) return
 * HC_ERR_TOO_LARGE before anything runs.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Its first call on a device looks the buffer's address up with that device
 * current; make that first call before any stream capture.  All calls share the
 * one buffer, which keeps the last call's contents: calls whose work overlaps on
 * the GPU (other streams, other threads) race on it and must be serialised by
 * the caller.
 */
int hc_pre_fused_noalloc(const float *x, const float *fn_w, const float *scale, const float *base,
                         int T, int s, int d, int iters, float eps,
                         float *pre, float *post, float *comb, float *y, void *stream);

/*
 * hc_post -- the post-branch half of a site (hyper.rs `post`):
 *   x_out[t, k, :] = post[t, k] * f[t, :] + sum_j comb[t, j, k] * x[t, j, :]
 * where x is the site's INPUT stream state (the residual), not the layer's.
 *   x [T, s, d] (in), f [T, d] branch output (in), post [T, s] (in),
 *   comb [T, s, s] (in), x_out [T, s, d] (out; must not overlap x, f, post or
 *   comb -- the pages ping-pong two state buffers and never update in place).
 */
int hc_post(const float *x, const float *f, const float *post, const float *comb,
            float *x_out, int T, int s, int d, void *stream);

/*
 * hc_rms_norm_q8 -- the branch input of a site (hyper.rs module header:
 * f = branch(rms_norm(y))), with the int8 pair the pages' fused v4z pre kernel
 * emits beside it:
 *   z[t, i] = y[t, i] * rsqrt(mean_i(y[t, :]^2) + eps_norm) * norm_w[i]
 *   per block of 32 consecutive z of a token (GGML Q8_0 layout; the pages give
 *   only the buffer shapes int8 [d] and float [d/32]):
 *     q_scale = amax / 127,  q = round-half-away(z * (1 / q_scale)), 0 if q_scale = 0
 *   y [T, d] (in), norm_w [d] (in), z [T, d] (out), q [T, d] int8 (out, optional),
 *   q_scale [T, d/32] (out, optional: q and q_scale are both given or both NULL).
 *   d % 4 == 0, and d % 32 == 0 when q is given; eps_norm >= 0 and finite.
 *   The int8 codes are decided in IEEE float32 (divide, reciprocal, multiply,
 *   round half away from zero) from the float32 z.
 */
int hc_rms_norm_q8(const float *y, const float *norm_w, int T, int d, float eps_norm,
                   float *z, signed char *q, float *q_scale, void *stream);

/*
 * hc_pre_fused_norm -- the pre-chain and the branch input f's norm, the pages' v4z
 * pre kernel (hc_fused_gate.rs page, the v4z arm: the rms_norm and its int8 / float
 * pair emitted by the pre kernel after the collapse): hc_pre_fused's outputs plus
 * hc_rms_norm_q8's z (and q, q_scale) of its y.  Arguments as for those two calls;
 * z, q and q_scale must not overlap any other argument.  Everything is validated
 * before anything is launched.
 * When the cluster path runs the shape and d / 16 is a multiple of 32 (e.g.
 * s <= 4, d = 4096) it can be ONE launch: each CTA of a cluster sends its share of
 * every token's sum of y^2 to the other fifteen, then writes z and the Q8_0 pair of
 * its own columns, so y is not read back by a second kernel.  Its sum of squares has
 * another fixed order than hc_rms_norm_q8's, so z may differ from the two-call result
 * in the last bits (still bit-identical run to run, and the same bits at any T).
 * hc_pre_fused_norm takes the one launch while the cluster path runs its one-tile
 * decode variant (up to 112 tokens at s = 4, d = 4096 on a GB300), where it is the
 * faster choice; for larger T, and for other shapes, it runs hc_pre_fused then
 * hc_rms_norm_q8 (at prefill sizes the persistent kernel's collapse warps, which
 * would also write z and the pair, are slower than a second launch over every SM).
 */
int hc_pre_fused_norm(const float *x, const float *fn_w, const float *scale, const float *base,
                      int T, int s, int d, int iters, float eps,
                      const float *norm_w, float eps_norm,
                      float *pre, float *post, float *comb, float *y,
                      float *z, signed char *q, float *q_scale,
                      void *workspace, size_t ws_bytes, void *stream);

/*
 * hc_pre_fused_norm with an explicit kernel path for the pre-chain (enum
 * hc_pre_path): HC_PATH_CLUSTER is one launch at any T where the shape allows it
 * (above), else the cluster pre-chain then hc_rms_norm_q8; the other paths are
 * always the two launches.
 */
int hc_pre_fused_norm_path(const float *x, const float *fn_w, const float *scale, const float *base,
                           int T, int s, int d, int iters, float eps,
                           const float *norm_w, float eps_norm,
                           float *pre, float *post, float *comb, float *y,
                           float *z, signed char *q, float *q_scale,
                           void *workspace, size_t ws_bytes, void *stream, int path);

/*
 * hc_post_pre_fused -- the boundary between two sites in one call: site i's
 * hc_post followed by site i+1's pre-chain on its result (hyper.rs module header:
 * the post formula, then the next site's "mixes", "mixes *= rsqrt", "sinkhorn"
 * and "y" lines; the pages' walk runs post_t1_ws -> pre_t1_ws back to back).
 *   x_prev [T, s, d]      site i's input state (in)
 *   f [T, d], post_prev [T, s], comb_prev [T, s, s]   site i's branch output and
 *                          gates (in)
 *   fn_w, scale, base     site i+1's trio, as for hc_pre_fused (in)
 *   x_new [T, s, d]       post_prev . f + comb_prev^T x_prev, the new state (out)
 *   pre, post, comb, y    site i+1's pre-chain outputs on x_new (out)
 * x_new is bit-identical to hc_post's output, and pre/post/comb/y to
 * hc_pre_fused on x_new, on the cluster path; there the new state is formed in
 * shared memory from one read of x_prev, so it is not read back from memory.
 * The cluster path takes the shapes hc_pre_fused's does with d <= 4096; shapes
 * the wide path takes run hc_post then the wide pre-chain (two launches, the
 * same bits as the two calls); other shapes run hc_post then the generic
 * pre-chain.  Outputs must not overlap any input or each other; workspace as
 * for hc_pre_fused, and outputs are valid only while hc_workspace_status reads
 * HC_OK (on the cluster path x_new too is left unwritten while it does not).
 */
int hc_post_pre_fused(const float *x_prev, const float *f, const float *post_prev,
                      const float *comb_prev, const float *fn_w, const float *scale,
                      const float *base, int T, int s, int d, int iters, float eps,
                      float *x_new, float *pre, float *post, float *comb, float *y,
                      void *workspace, size_t ws_bytes, void *stream);

/* hc_post_pre_fused with an explicit kernel path (enum hc_pre_path). */
int hc_post_pre_fused_path(const float *x_prev, const float *f, const float *post_prev,
                           const float *comb_prev, const float *fn_w, const float *scale,
                           const float *base, int T, int s, int d, int iters, float eps,
                           float *x_new, float *pre, float *post, float *comb, float *y,
                           void *workspace, size_t ws_bytes, void *stream, int path);

/*
 * hc_head -- gated-head trunk exit [T, s, d] -> [T, d] (hyper.rs `collapse`, case
 * HcCollapse::GatedHead: the head trio of HyperHead::load -- fn_w with rows equal
 * to the streams, base [s] and ONE scale -- then rowsq_scale, hc_head_pre and
 * hc_collapse).  Per token:
 *   mixes[c] = rsqrt(mean(x[t]^2) + eps) * (fn_w[c, :] . x[t, :, :])   c < s
 *   gate[c]  = sigmoid(mixes[c] * scale[0] + base[c]) + eps
 *   y[t, :]  = sum_c gate[c] * x[t, c, :]
 * The pages print no formula for the head gates; the one above is the site's pre
 * gate with the head's single scale.
 *   x [T, s, d] (in), fn_w [s, s*d] row-major (in), scale [1] (in), base [s] (in),
 *   gates [T, s] (out, optional: NULL skips it), y [T, d] (out),
 *   workspace, ws_bytes: >= hc_pre_workspace_bytes(T, s, d), as for hc_pre_fused.
 * Same conventions, limits, determinism and batch invariance (cluster path) as
 * hc_pre_fused; the cluster path takes the shapes it takes there, the wide path
 * has no head variant (HC_ERR_UNSUPPORTED; HC_PATH_AUTO runs the generic path
 * for s > 4).
 */
int hc_head(const float *x, const float *fn_w, const float *scale, const float *base,
            int T, int s, int d, float eps, float *gates, float *y,
            void *workspace, size_t ws_bytes, void *stream);

/* hc_head with an explicit kernel path (enum hc_pre_path). */
int hc_head_path(const float *x, const float *fn_w, const float *scale, const float *base,
                 int T, int s, int d, float eps, float *gates, float *y,
                 void *workspace, size_t ws_bytes, void *stream, int path);

/*
 * hc_mean -- unweighted stream mean [T, s, d] -> [T, d] (hyper.rs
 * `contract_mean`, the glm5_next trunk exit `HcCollapse::Mean`).
 *   x [T, s, d] (in), out [T, d] (out, must not overlap x).
 */
int hc_mean(const float *x, float *out, int T, int s, int d, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_GB300_HC_H */
