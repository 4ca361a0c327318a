// hc_internal.cuh -- private declarations shared by the library's translation units.
//
// Nothing here is part of the C ABI (include/hc.h is).  The library is written
// for sm_103a only: it is compiled with -gencode arch=compute_103a,code=sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "hc.h"

namespace hc {

// ---------------------------------------------------------------- workspace status block
// The first kStatusBytes of every hc_pre_fused workspace hold a status block.
// Kernels only ever write a non-zero code into it (first error wins); the host
// clears it with hc_workspace_init and reads it with hc_workspace_status.
constexpr size_t kStatusBytes = 256;
struct StatusBlock {
    unsigned int code;    // 0 = ok, else a DevErr value
    unsigned int where;   // kernel-specific location of the first error
    unsigned int block;   // linear block index that reported it
    unsigned int pad[61];
};
static_assert(sizeof(StatusBlock) == kStatusBytes, "status block is 256 bytes");

// ---------------------------------------------------------------- phase stamps
// A build with -DHC_STAMPS (build.build(stamps=True), a separate library) makes the
// cluster and wide pre kernels write %globaltimer at phase boundaries of every tile into
// the workspace, right after the status block: [kStampCtas][kStampTiles][kStampEvents]
// 64-bit nanosecond stamps.  Cluster kernel: CTAs 0 and 8 of cluster 0 (the owners of
// tokens 0 and 8 of every tile).  Wide kernel: slot 0 CTA 0's own phases, slot 1 the
// reduction of column 0 and the finish of every tile, by whichever CTA did them.  Stamps
// of tiles beyond kStampTiles are dropped.
constexpr int kStampCtas = 2, kStampTiles = 512, kStampEvents = 16;
constexpr size_t kStampBytes = (size_t)kStampCtas * kStampTiles * kStampEvents * 8;
enum StampEvent : int {
    kEvStageReady = 0,   // compute warpgroup 0: the tile's stage is ready
    kEvDotsDone,         // compute warpgroup 0: dots and squares done (thread 0)
    kEvShipped,          // compute warpgroup 0: partials shipped (thread 0)
    kEvPartials,         // finisher: every partial of the owned token arrived
    kEvGatesSent,        // finisher: pre sent to every CTA
    kEvPreArrived,       // collapse: the tile's pre gates are all in
    kEvCollapsed,        // collapse: y written
    kEvRefilled,         // collapse: the stage's next load issued
    kEvXfStart,          // fused: transform of the tile begins (collapse warps)
    kEvXfLanded,         // fused: the tile's stage and f slice have landed
    kEvXfDone,           // fused: x' stored, stage released to the compute warps
    kEvSinkDone,         // Sinkhorn warp: the tile's comb blocks written
    kEvKernelStart,      // (tile 0 only) kernel entry
};
#ifdef HC_STAMPS
constexpr size_t kWorkspaceExtra = kStampBytes;
#else
constexpr size_t kWorkspaceExtra = 0;
#endif

enum DevErr : unsigned int {
    kDevOk = 0,
    kDevWaitTimeout = 1,   // a bounded wait on an mbarrier gave up
    kDevBounds = 2,        // (bounds-checked build) a store fell outside its buffer and was skipped
};

__device__ __forceinline__ void report_error(StatusBlock *sb, unsigned int code, unsigned int where)
{
    if (sb != nullptr && atomicCAS(&sb->code, 0u, code) == 0u) {
        sb->where = where;
        sb->block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    }
}

// ---------------------------------------------------------------- bounds-checked stores
// A build with -DHC_DEBUG_BOUNDS (build.build(bounds=True), a separate library) checks the
// plain global stores of the cluster, helper and wide kernels (y, pre, post, comb and the
// helper's partials) against the number of elements of the buffer each writes: a store at or past the
// end is not performed, and the kernel reports kDevBounds with the store's site (below) in
// the status word.  Any other build stores unconditionally (the same code as a plain store).
enum StoreSite : unsigned int { kStoreY = 100, kStorePre, kStorePost, kStoreComb, kStorePart };

template <typename T>
__device__ __forceinline__ void store_checked(T *base, size_t i, size_t n, const T &v, StatusBlock *sb,
                                              unsigned int site)
{
#ifdef HC_DEBUG_BOUNDS
    if (i >= n) {
        report_error(sb, kDevBounds, site);
        return;
    }
#else
    (void)n;
    (void)sb;
    (void)site;
#endif
    base[i] = v;
}

// ---------------------------------------------------------------- device properties (host)
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};
// Cached per device; returns false if the CUDA runtime fails.
bool device_info(DeviceInfo &out);

// Unique id (cuCtxGetId) of the CUDA context current on the calling thread, 0 if none
// is current yet.  Per-device set-up (function attributes, symbol addresses) is cached
// under it, so a device reset, which replaces the context, makes the set-up run again.
// A float32 tensor map (no interleave or swizzle, 256-byte L2 promotion, zero fill
// out of bounds, unit element strides) of `rank` dimensions: dims[rank], byte strides of
// dimensions 1.. (strides[rank-1]), box[rank].  A map depends on nothing but these
// arguments, so maps are kept in a small table keyed on them and repeated calls on the
// same buffers and shapes skip the encoder.  False if the encoder is missing or refuses.
bool tensor_map_f32(CUtensorMap *out, int rank, const void *base, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box);

unsigned long long context_id();

// ---------------------------------------------------------------- launchers (host)
// All launchers assume validated arguments and return a cudaError_t.
cudaError_t launch_post(const float *x, const float *f, const float *post, const float *comb,
                        float *x_out, int T, int s, int d, cudaStream_t st);
cudaError_t launch_expand(const float *emb, float *x, int T, int s, int d, cudaStream_t st);
cudaError_t launch_mean(const float *x, float *out, int T, int s, int d, cudaStream_t st);
// Branch-input norm z = y * rsqrt(mean(y^2) + eps_norm) * norm_w, and optionally its
// Q8_0 pair (q [T, d] int8, q_scale [T, d/32]); q == nullptr skips the pair.
cudaError_t launch_rms_norm_q8(const float *y, const float *norm_w, int T, int d, float eps_norm, float *z,
                               signed char *q, float *q_scale, cudaStream_t st);

// Generic pre path: split-K mixes partials, then a per-token finish + collapse.
size_t generic_workspace_bytes(int T, int s, int d);
cudaError_t launch_pre_generic(const float *x, const float *fn_w, const float *scale,
                               const float *base, int T, int s, int d, int iters, float eps,
                               float *pre, float *post, float *comb, float *y,
                               void *workspace, cudaStream_t st);

// Wide-stream pre path (5 <= s <= 8): one persistent whole-GPU launch, every CTA a fixed
// K slice of fn_w in TMEM; wide_supported() says whether the shape has a balanced split
// and the device can run it.
size_t wide_workspace_bytes(int T, int s, int d);
bool wide_supported(int s, int d);
cudaError_t launch_pre_wide(const float *x, const float *fn_w, const float *scale, const float *base,
                            int T, int s, int d, int iters, float eps, float *pre, float *post,
                            float *comb, float *y, void *workspace, cudaStream_t st);

// Cluster pre path (one fused launch).  cluster_supported() says whether the
// shape fits and the device can co-schedule the clusters.
bool cluster_shape_ok(int s, int d);
bool cluster_supported(int s, int d);
bool cluster_supported(int s, int d, bool head);
bool cluster_fused_supported(int s, int d);   // fused post -> pre: also d / 16 <= 256
bool cluster_norm_supported(int s, int d);    // pre + branch-input norm: also (d / 16) % 32 == 0
// Tokens up to which the cluster path runs its one-tile (decode) variant for this shape (0 if
// the norm cannot run in it): there the pre-chain and norm in one launch are the faster
// choice; above it the persistent variant's collapse warps make two launches faster.
int cluster_decode_tokens(int s, int d);
// The pre-chain and the branch-input norm (z, and the Q8_0 pair when q is given) in one
// launch of the cluster kernel.
cudaError_t launch_pre_norm_cluster(const float *x, const float *fn_w, const float *scale,
                                    const float *base, int T, int s, int d, int iters, float eps,
                                    const float *norm_w, float eps_norm, float *pre, float *post, float *comb,
                                    float *y, float *z, signed char *q, float *q_scale, void *workspace,
                                    cudaStream_t st);
// At prefill sizes the cluster kernel's launch is followed by the helper kernel, on the SMs
// the clusters leave free, for the batch's last tokens, when ws_bytes holds its partials
// (cluster_helper_workspace_bytes; the same bits either way).
size_t cluster_helper_workspace_bytes(int T, int s, int d);
// Tokens the helper kernel takes from the end of a batch (0: the cluster kernel alone).
int cluster_helper_tokens(int T, int s, int d, bool fused, size_t ws_bytes);
cudaError_t launch_pre_cluster(const float *x, const float *fn_w, const float *scale,
                               const float *base, int T, int s, int d, int iters, float eps,
                               float *pre, float *post, float *comb, float *y,
                               void *workspace, size_t ws_bytes, cudaStream_t st);

// Fused post -> pre: x_new = post_prev . f + comb_prev^T x_prev, then the pre-chain of
// the next site on x_new, in one launch of the cluster kernel.
cudaError_t launch_post_pre_cluster(const float *x_prev, const float *f, const float *post_prev,
                                    const float *comb_prev, const float *fn_w, const float *scale,
                                    const float *base, int T, int s, int d, int iters, float eps,
                                    float *x_new, float *pre, float *post, float *comb, float *y,
                                    void *workspace, size_t ws_bytes, cudaStream_t st);

// Gated-head trunk exit: rows = streams, one scale, gates (optional output) + collapse.
cudaError_t launch_head_cluster(const float *x, const float *fn_w, const float *scale,
                                const float *base, int T, int s, int d, float eps, float *gates,
                                float *y, void *workspace, cudaStream_t st);
cudaError_t launch_head_generic(const float *x, const float *fn_w, const float *scale,
                                const float *base, int T, int s, int d, float eps, float *gates,
                                float *y, void *workspace, cudaStream_t st);

}  // namespace hc
