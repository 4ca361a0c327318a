// hc_api.cu -- the extern "C" entry points declared in include/hc.h.
//
// Every entry validates its arguments on the host before enqueuing anything
// (the pages refuse bad shapes loudly by name -- hyper.rs HyperTopology::from_plan
// and load_site -- and here a status code plays that role), then calls the
// launcher of the chosen kernel path and reports the launch's cudaError.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "hc_internal.cuh"

namespace hc {

unsigned long long context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
        cudaGetLastError();
    });
    if (!get_current || !get_id)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

namespace {

struct TmapKey {
    const void *base;
    int rank;
    cuuint64_t dims[5];
    cuuint64_t strides[4];
    cuuint32_t box[5];
};

struct TmapEntry {
    bool used = false;
    TmapKey key;
    CUtensorMap map;
};

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder()
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

}  // namespace

bool tensor_map_f32(CUtensorMap *out, int rank, const void *base, const cuuint64_t *dims,
                    const cuuint64_t *strides, const cuuint32_t *box)
{
    constexpr int kEntries = 32;
    static std::mutex mu;
    static TmapEntry table[kEntries];
    static int next = 0;
    if (rank < 1 || rank > 5)
        return false;
    TmapKey key;
    memset(&key, 0, sizeof(key));
    key.base = base;
    key.rank = rank;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank)
            key.strides[i] = strides[i];
    }
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int e = 0; e < kEntries; ++e)
            if (table[e].used && memcmp(&table[e].key, &key, sizeof(key)) == 0) {
                *out = table[e].map;
                return true;
            }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = tmap_encoder();
    if (!enc)
        return false;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (enc(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    TmapEntry &slot = table[next];
    next = (next + 1) % kEntries;
    slot.used = true;
    slot.key = key;
    slot.map = *out;
    return true;
}

bool device_info(DeviceInfo &out)
{
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &c = cache[dev];
    if (c.device != dev) {
        DeviceInfo n;
        n.device = dev;
        if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return false;
        c = n;
    }
    out = c;
    return true;
}

}  // namespace hc

namespace {

using hc::kStatusBytes;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Byte ranges [a, a+na) and [b, b+nb) overlap (empty ranges never do).
bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    if (na == 0 || nb == 0)
        return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool dims_ok(int T, int s, int d)
{
    if (T < 0 || s < 1 || s > 8 || d < 4)
        return false;
    const int64_t n = (int64_t)T * s * d;
    return n < ((int64_t)1 << 31);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? HC_OK : HC_ERR_CUDA; }

// Workspace bytes the given (resolved) kernel path needs; hc_pre_workspace_bytes is the
// largest over the paths, so a workspace of that size serves any of them.
size_t path_workspace_bytes(int path, int T, int s, int d)
{
    const size_t status = kStatusBytes + hc::kWorkspaceExtra;
    size_t need = status;
    if (path == HC_PATH_GENERIC)
        need = hc::generic_workspace_bytes(T, s, d);
    else if (path == HC_PATH_WIDE)
        need = hc::wide_workspace_bytes(T, s, d);
    return need > status ? need : status;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char *hc_status_string(int rc)
{
    switch (rc) {
    case HC_OK: return "ok";
    case HC_ERR_NULL: return "a required pointer is NULL";
    case HC_ERR_DIM: return "dimension or parameter out of range (need T >= 0, 1 <= s <= 8, d >= 4, T*s*d < 2^31, iters >= 1, finite eps > 0)";
    case HC_ERR_ALIGN: return "misaligned pointer or d not a multiple of 4 (tensors 16-byte aligned, gates 4-byte)";
    case HC_ERR_ALIAS: return "an output buffer overlaps an input or another output";
    case HC_ERR_WORKSPACE: return "workspace is NULL, misaligned or smaller than hc_pre_workspace_bytes";
    case HC_ERR_CUDA: return "the CUDA runtime reported an error";
    case HC_ERR_DEVICE: return "a kernel flagged an error in the workspace status word (bounded wait gave up)";
    case HC_ERR_UNSUPPORTED: return "the requested kernel path cannot run this shape on this device";
    case HC_ERR_TOO_LARGE: return "shape needs more scratch than hc_pre_fused_noalloc's 4 MiB static buffer holds";
    default: return "unknown status";
    }
}

int hc_expand(const float *emb, float *x, int T, int s, int d, void *stream)
{
    if (!dims_ok(T, s, d))
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!emb || !x)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(emb, 16) || !aligned(x, 16))
        return HC_ERR_ALIGN;
    const size_t in_b = (size_t)T * d * 4, out_b = in_b * s;
    if (overlap(emb, in_b, x, out_b))
        return HC_ERR_ALIAS;
    return cuda_rc(hc::launch_expand(emb, x, T, s, d, as_stream(stream)));
}

int hc_mean(const float *x, float *out, int T, int s, int d, void *stream)
{
    if (!dims_ok(T, s, d))
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!x || !out)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(x, 16) || !aligned(out, 16))
        return HC_ERR_ALIGN;
    const size_t out_b = (size_t)T * d * 4, in_b = out_b * s;
    if (overlap(x, in_b, out, out_b))
        return HC_ERR_ALIAS;
    return cuda_rc(hc::launch_mean(x, out, T, s, d, as_stream(stream)));
}

int hc_post(const float *x, const float *f, const float *post, const float *comb, float *x_out,
            int T, int s, int d, void *stream)
{
    if (!dims_ok(T, s, d))
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!x || !f || !post || !comb || !x_out)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(x, 16) || !aligned(f, 16) || !aligned(x_out, 16) || !aligned(post, 4) ||
        !aligned(comb, 4))
        return HC_ERR_ALIGN;
    const size_t xb = (size_t)T * s * d * 4, fb = (size_t)T * d * 4;
    const size_t pb = (size_t)T * s * 4, cb = (size_t)T * s * s * 4;
    if (overlap(x_out, xb, x, xb) || overlap(x_out, xb, f, fb) || overlap(x_out, xb, post, pb) ||
        overlap(x_out, xb, comb, cb))
        return HC_ERR_ALIAS;
    return cuda_rc(hc::launch_post(x, f, post, comb, x_out, T, s, d, as_stream(stream)));
}

size_t hc_pre_workspace_bytes(int T, int s, int d)
{
    if (!dims_ok(T, s, d))
        return 0;
    // Any path may be asked for, so size for the larger of the two (a phase-stamp build
    // keeps its stamps after the status block).
    const size_t g = hc::generic_workspace_bytes(T, s, d);
    const size_t c0 = kStatusBytes + hc::kWorkspaceExtra, ch = hc::cluster_helper_workspace_bytes(T, s, d);
    const size_t c = c0 > ch ? c0 : ch;
    const size_t w = hc::wide_workspace_bytes(T, s, d);
    const size_t m = g > c ? g : c;
    return m > w ? m : w;
}

int hc_workspace_init(void *workspace, size_t ws_bytes, void *stream)
{
    if (!workspace)
        return HC_ERR_NULL;
    return cuda_rc(cudaMemsetAsync(workspace, 0, ws_bytes, as_stream(stream)));
}

int hc_workspace_status(const void *workspace, void *stream)
{
    if (!workspace)
        return HC_ERR_NULL;
    unsigned int code = 0;
    cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost,
                                    as_stream(stream));
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess)
        return HC_ERR_CUDA;
    return code == 0 ? HC_OK : HC_ERR_DEVICE;
}

int hc_pre_auto_path(int T, int s, int d)
{
    (void)T;
    if (!dims_ok(T, s, d) || d % 4)
        return HC_PATH_GENERIC;
    if (hc::cluster_supported(s, d))
        return HC_PATH_CLUSTER;
    return hc::wide_supported(s, d) ? HC_PATH_WIDE : HC_PATH_GENERIC;
}

int hc_pre_helper_tokens(int T, int s, int d, int fused, size_t ws_bytes)
{
    if (!dims_ok(T, s, d))
        return -1;
    if (d % 4 || T == 0 || !hc::cluster_supported(s, d))
        return 0;
    return hc::cluster_helper_tokens(T, s, d, fused != 0, ws_bytes);
}

}  // extern "C"

namespace {

// Every check of hc_pre_fused_path, with HC_PATH_AUTO resolved into `path`; HC_OK (with
// nothing to run when T == 0) or the status to return.
int pre_checks(const float *x, const float *fn_w, const float *scale, const float *base, int T, int s, int d,
               int iters, float eps, float *pre, float *post, float *comb, float *y, void *workspace,
               size_t ws_bytes, int &path)
{
    if (!dims_ok(T, s, d) || iters < 1 || !(eps > 0.f) || !std::isfinite(eps))
        return HC_ERR_DIM;
    if (path != HC_PATH_AUTO && path != HC_PATH_GENERIC && path != HC_PATH_CLUSTER && path != HC_PATH_WIDE)
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!x || !fn_w || !scale || !base || !pre || !post || !comb || !y)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(x, 16) || !aligned(fn_w, 16) || !aligned(y, 16) || !aligned(scale, 4) ||
        !aligned(base, 4) || !aligned(pre, 4) || !aligned(post, 4) || !aligned(comb, 4))
        return HC_ERR_ALIGN;
    const int R = (2 + s) * s;
    const size_t xb = (size_t)T * s * d * 4, wb = (size_t)R * s * d * 4;
    const size_t gb = (size_t)T * s * 4, cb = (size_t)T * s * s * 4, yb = (size_t)T * d * 4;
    const void *ins[4] = {x, fn_w, scale, base};
    const size_t in_b[4] = {xb, wb, 12, (size_t)R * 4};
    const void *outs[4] = {pre, post, comb, y};
    const size_t out_b[4] = {gb, gb, cb, yb};
    for (int o = 0; o < 4; ++o) {
        for (int i = 0; i < 4; ++i)
            if (overlap(outs[o], out_b[o], ins[i], in_b[i]))
                return HC_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 4; ++o2)
            if (overlap(outs[o], out_b[o], outs[o2], out_b[o2]))
                return HC_ERR_ALIAS;
    }
    if (path == HC_PATH_AUTO)
        path = hc_pre_auto_path(T, s, d);
    if (!workspace || !aligned(workspace, 16) || ws_bytes < path_workspace_bytes(path, T, s, d))
        return HC_ERR_WORKSPACE;
    for (int o = 0; o < 4; ++o)
        if (overlap(outs[o], out_b[o], workspace, ws_bytes))
            return HC_ERR_ALIAS;
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_b[i], workspace, ws_bytes))
            return HC_ERR_ALIAS;
    return HC_OK;
}

}  // namespace

extern "C" {

int hc_pre_fused_path(const float *x, const float *fn_w, const float *scale, const float *base,
                      int T, int s, int d, int iters, float eps, float *pre, float *post,
                      float *comb, float *y, void *workspace, size_t ws_bytes, void *stream, int path)
{
    const int rc = pre_checks(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y, workspace, ws_bytes,
                              path);
    if (rc != HC_OK || T == 0)
        return rc;
    cudaStream_t st = as_stream(stream);
    if (path == HC_PATH_CLUSTER) {
        if (!hc::cluster_supported(s, d))
            return HC_ERR_UNSUPPORTED;
        return cuda_rc(hc::launch_pre_cluster(x, fn_w, scale, base, T, s, d, iters, eps, pre, post,
                                              comb, y, workspace, ws_bytes, st));
    }
    if (path == HC_PATH_WIDE) {
        if (!hc::wide_supported(s, d))
            return HC_ERR_UNSUPPORTED;
        return cuda_rc(hc::launch_pre_wide(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb,
                                           y, workspace, st));
    }
    return cuda_rc(hc::launch_pre_generic(x, fn_w, scale, base, T, s, d, iters, eps, pre, post,
                                          comb, y, workspace, st));
}

int hc_rms_norm_q8(const float *y, const float *norm_w, int T, int d, float eps_norm, float *z,
                   signed char *q, float *q_scale, void *stream)
{
    if (T < 0 || d < 4 || !(eps_norm >= 0.f) || !std::isfinite(eps_norm) || (int64_t)T * d >= ((int64_t)1 << 31))
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!y || !norm_w || !z || (!q) != (!q_scale))
        return HC_ERR_NULL;
    if (d % 4 || (q && d % 32) || !aligned(y, 16) || !aligned(norm_w, 16) || !aligned(z, 16) ||
        (q && (!aligned(q, 4) || !aligned(q_scale, 4))))
        return HC_ERR_ALIGN;
    const size_t yb = (size_t)T * d * 4, qb = q ? (size_t)T * d : 0, sb = q ? (size_t)T * (d / 32) * 4 : 0;
    const void *ins[2] = {y, norm_w};
    const size_t in_b[2] = {yb, (size_t)d * 4};
    const void *outs[3] = {z, q, q_scale};
    const size_t out_b[3] = {yb, qb, sb};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 2; ++i)
            if (overlap(outs[o], out_b[o], ins[i], in_b[i]))
                return HC_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 3; ++o2)
            if (overlap(outs[o], out_b[o], outs[o2], out_b[o2]))
                return HC_ERR_ALIAS;
    }
    return cuda_rc(hc::launch_rms_norm_q8(y, norm_w, T, d, eps_norm, z, q, q_scale, as_stream(stream)));
}

int hc_pre_fused_norm_path(const float *x, const float *fn_w, const float *scale, const float *base, int T,
                           int s, int d, int iters, float eps, const float *norm_w, float eps_norm, float *pre,
                           float *post, float *comb, float *y, float *z, signed char *q, float *q_scale,
                           void *workspace, size_t ws_bytes, void *stream, int path)
{
    // Every argument is checked before anything is launched: the pre-chain's (which also
    // bound T, s and d), then the norm's.
    if (!(eps_norm >= 0.f) || !std::isfinite(eps_norm))
        return HC_ERR_DIM;
    const int asked = path;
    const int rc = pre_checks(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y, workspace, ws_bytes,
                              path);
    if (rc != HC_OK || T == 0)
        return rc;
    {
        if (!norm_w || !z || (!q) != (!q_scale))
            return HC_ERR_NULL;
        if ((q && d % 32) || !aligned(norm_w, 16) || !aligned(z, 16) ||
            (q && (!aligned(q, 4) || !aligned(q_scale, 4))))
            return HC_ERR_ALIGN;
        const int R = (2 + s) * s;
        const size_t xb = (size_t)T * s * d * 4, yb = (size_t)T * d * 4;
        const size_t qb = q ? (size_t)T * d : 0, sb = q ? (size_t)T * (d / 32) * 4 : 0;
        const void *others[9] = {x, fn_w, scale, base, pre, post, comb, y, workspace};
        const size_t other_b[9] = {xb, (size_t)R * s * d * 4, 12, (size_t)R * 4, (size_t)T * s * 4,
                                   (size_t)T * s * 4, (size_t)T * s * s * 4, yb, ws_bytes};
        const void *outs[3] = {z, q, q_scale};
        const size_t out_b[3] = {yb, qb, sb};
        for (int o = 0; o < 3; ++o) {
            for (int i = 0; i < 9; ++i)
                if (overlap(outs[o], out_b[o], others[i], other_b[i]))
                    return HC_ERR_ALIAS;
            if (overlap(outs[o], out_b[o], norm_w, (size_t)d * 4))
                return HC_ERR_ALIAS;
            for (int o2 = o + 1; o2 < 3; ++o2)
                if (overlap(outs[o], out_b[o], outs[o2], out_b[o2]))
                    return HC_ERR_ALIAS;
        }
    }
    cudaStream_t st = as_stream(stream);
    // One launch when the cluster path runs the shape and its slices hold whole Q8_0 blocks:
    // always when that path was asked for, and under HC_PATH_AUTO while the decode variant
    // runs (above that size the persistent kernel's collapse warps, which would also write
    // z and the pair, are slower than a second, whole-GPU norm launch).
    if (path == HC_PATH_CLUSTER && hc::cluster_norm_supported(s, d) &&
        (asked == HC_PATH_CLUSTER || T <= hc::cluster_decode_tokens(s, d)))
        return cuda_rc(hc::launch_pre_norm_cluster(x, fn_w, scale, base, T, s, d, iters, eps, norm_w, eps_norm, pre,
                                                   post, comb, y, z, q, q_scale, workspace, st));
    if (asked == HC_PATH_CLUSTER && !hc::cluster_supported(s, d))
        return HC_ERR_UNSUPPORTED;
    const int rc2 = hc_pre_fused_path(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y, workspace,
                                      ws_bytes, stream, path);
    if (rc2 != HC_OK)
        return rc2;
    return hc_rms_norm_q8(y, norm_w, T, d, eps_norm, z, q, q_scale, stream);
}

int hc_pre_fused_norm(const float *x, const float *fn_w, const float *scale, const float *base, int T, int s,
                      int d, int iters, float eps, const float *norm_w, float eps_norm, float *pre, float *post,
                      float *comb, float *y, float *z, signed char *q, float *q_scale, void *workspace,
                      size_t ws_bytes, void *stream)
{
    return hc_pre_fused_norm_path(x, fn_w, scale, base, T, s, d, iters, eps, norm_w, eps_norm, pre, post, comb, y,
                                  z, q, q_scale, workspace, ws_bytes, stream, HC_PATH_AUTO);
}

int hc_post_pre_fused_path(const float *x_prev, const float *f, const float *post_prev,
                           const float *comb_prev, const float *fn_w, const float *scale,
                           const float *base, int T, int s, int d, int iters, float eps, float *x_new,
                           float *pre, float *post, float *comb, float *y, void *workspace,
                           size_t ws_bytes, void *stream, int path)
{
    if (!dims_ok(T, s, d) || iters < 1 || !(eps > 0.f) || !std::isfinite(eps))
        return HC_ERR_DIM;
    if (path != HC_PATH_AUTO && path != HC_PATH_GENERIC && path != HC_PATH_CLUSTER && path != HC_PATH_WIDE)
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (!x_prev || !f || !post_prev || !comb_prev || !fn_w || !scale || !base || !x_new || !pre ||
        !post || !comb || !y)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(x_prev, 16) || !aligned(f, 16) || !aligned(x_new, 16) || !aligned(fn_w, 16) ||
        !aligned(y, 16) || !aligned(post_prev, 4) || !aligned(comb_prev, 4) || !aligned(scale, 4) ||
        !aligned(base, 4) || !aligned(pre, 4) || !aligned(post, 4) || !aligned(comb, 4))
        return HC_ERR_ALIGN;
    const int R = (2 + s) * s;
    const size_t xb = (size_t)T * s * d * 4, fb = (size_t)T * d * 4, wb = (size_t)R * s * d * 4;
    const size_t gb = (size_t)T * s * 4, cb = (size_t)T * s * s * 4;
    const void *ins[7] = {x_prev, f, post_prev, comb_prev, fn_w, scale, base};
    const size_t in_b[7] = {xb, fb, gb, cb, wb, 12, (size_t)R * 4};
    const void *outs[5] = {x_new, pre, post, comb, y};
    const size_t out_b[5] = {xb, gb, gb, cb, fb};
    for (int o = 0; o < 5; ++o) {
        for (int i = 0; i < 7; ++i)
            if (overlap(outs[o], out_b[o], ins[i], in_b[i]))
                return HC_ERR_ALIAS;
        for (int o2 = o + 1; o2 < 5; ++o2)
            if (overlap(outs[o], out_b[o], outs[o2], out_b[o2]))
                return HC_ERR_ALIAS;
    }
    if (path == HC_PATH_AUTO) {
        path = hc::cluster_fused_supported(s, d) ? HC_PATH_CLUSTER
                                                  : (hc::wide_supported(s, d) ? HC_PATH_WIDE : HC_PATH_GENERIC);
    }
    if (!workspace || !aligned(workspace, 16) || ws_bytes < path_workspace_bytes(path, T, s, d))
        return HC_ERR_WORKSPACE;
    for (int o = 0; o < 5; ++o)
        if (overlap(outs[o], out_b[o], workspace, ws_bytes))
            return HC_ERR_ALIAS;
    for (int i = 0; i < 7; ++i)
        if (overlap(ins[i], in_b[i], workspace, ws_bytes))
            return HC_ERR_ALIAS;

    cudaStream_t st = as_stream(stream);
    if (path == HC_PATH_CLUSTER) {
        if (!hc::cluster_fused_supported(s, d))
            return HC_ERR_UNSUPPORTED;
        return cuda_rc(hc::launch_post_pre_cluster(x_prev, f, post_prev, comb_prev, fn_w, scale, base, T, s, d,
                                                   iters, eps, x_new, pre, post, comb, y, workspace, ws_bytes, st));
    }
    if (path == HC_PATH_WIDE && !hc::wide_supported(s, d))
        return HC_ERR_UNSUPPORTED;
    // Shapes the fused kernel does not take: hc_post, then the pre-chain (wide or generic
    // path) on its output.
    const cudaError_t e = hc::launch_post(x_prev, f, post_prev, comb_prev, x_new, T, s, d, st);
    if (e != cudaSuccess)
        return HC_ERR_CUDA;
    if (path == HC_PATH_WIDE)
        return cuda_rc(hc::launch_pre_wide(x_new, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y,
                                           workspace, st));
    return cuda_rc(hc::launch_pre_generic(x_new, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y,
                                          workspace, st));
}

int hc_post_pre_fused(const float *x_prev, const float *f, const float *post_prev, const float *comb_prev,
                      const float *fn_w, const float *scale, const float *base, int T, int s, int d,
                      int iters, float eps, float *x_new, float *pre, float *post, float *comb, float *y,
                      void *workspace, size_t ws_bytes, void *stream)
{
    return hc_post_pre_fused_path(x_prev, f, post_prev, comb_prev, fn_w, scale, base, T, s, d, iters, eps,
                                  x_new, pre, post, comb, y, workspace, ws_bytes, stream, HC_PATH_AUTO);
}

int hc_head_path(const float *x, const float *fn_w, const float *scale, const float *base, int T,
                 int s, int d, float eps, float *gates, float *y, void *workspace, size_t ws_bytes,
                 void *stream, int path)
{
    if (!dims_ok(T, s, d) || !(eps > 0.f) || !std::isfinite(eps))
        return HC_ERR_DIM;
    if (path != HC_PATH_AUTO && path != HC_PATH_GENERIC && path != HC_PATH_CLUSTER && path != HC_PATH_WIDE)
        return HC_ERR_DIM;
    if (T == 0)
        return HC_OK;
    if (path == HC_PATH_WIDE)
        return HC_ERR_UNSUPPORTED;   // the gated head has no wide-stream kernel
    if (!x || !fn_w || !scale || !base || !y)
        return HC_ERR_NULL;
    if (d % 4 || !aligned(x, 16) || !aligned(fn_w, 16) || !aligned(y, 16) || !aligned(scale, 4) ||
        !aligned(base, 4) || (gates && !aligned(gates, 4)))
        return HC_ERR_ALIGN;
    const size_t xb = (size_t)T * s * d * 4, wb = (size_t)s * s * d * 4;
    const size_t gb = gates ? (size_t)T * s * 4 : 0, yb = (size_t)T * d * 4;
    const void *ins[4] = {x, fn_w, scale, base};
    const size_t in_b[4] = {xb, wb, 4, (size_t)s * 4};
    const void *outs[2] = {gates, y};
    const size_t out_b[2] = {gb, yb};
    for (int o = 0; o < 2; ++o)
        for (int i = 0; i < 4; ++i)
            if (overlap(outs[o], out_b[o], ins[i], in_b[i]))
                return HC_ERR_ALIAS;
    if (overlap(gates, gb, y, yb))
        return HC_ERR_ALIAS;
    if (path == HC_PATH_AUTO)
        path = hc::cluster_supported(s, d, true) ? HC_PATH_CLUSTER : HC_PATH_GENERIC;
    if (!workspace || !aligned(workspace, 16) || ws_bytes < path_workspace_bytes(path, T, s, d))
        return HC_ERR_WORKSPACE;
    for (int o = 0; o < 2; ++o)
        if (overlap(outs[o], out_b[o], workspace, ws_bytes))
            return HC_ERR_ALIAS;
    for (int i = 0; i < 4; ++i)
        if (overlap(ins[i], in_b[i], workspace, ws_bytes))
            return HC_ERR_ALIAS;

    cudaStream_t st = as_stream(stream);
    if (path == HC_PATH_CLUSTER) {
        if (!hc::cluster_supported(s, d, true))
            return HC_ERR_UNSUPPORTED;
        return cuda_rc(hc::launch_head_cluster(x, fn_w, scale, base, T, s, d, eps, gates, y, workspace, st));
    }
    return cuda_rc(hc::launch_head_generic(x, fn_w, scale, base, T, s, d, eps, gates, y, workspace, st));
}

int hc_head(const float *x, const float *fn_w, const float *scale, const float *base, int T, int s,
            int d, float eps, float *gates, float *y, void *workspace, size_t ws_bytes, void *stream)
{
    return hc_head_path(x, fn_w, scale, base, T, s, d, eps, gates, y, workspace, ws_bytes, stream,
                        HC_PATH_AUTO);
}

int hc_pre_fused(const float *x, const float *fn_w, const float *scale, const float *base, int T,
                 int s, int d, int iters, float eps, float *pre, float *post, float *comb, float *y,
                 void *workspace, size_t ws_bytes, void *stream)
{
    return hc_pre_fused_path(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y,
                             workspace, ws_bytes, stream, HC_PATH_AUTO);
}

}  // extern "C"
