// hc_noalloc.cu -- hc_pre_fused_noalloc: the pre-chain without any device allocation.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run a site.  A serving engine that carves all device memory into a fixed
// arena at start-up has nothing left for a cudaMalloc later; a plugin hosted by
// a framework that owns every allocation is not allowed to make one; and a
// latency-critical loop cannot afford cudaMalloc/cudaFree, which may block or
// synchronise the device.  hc_pre_fused needs a caller-supplied workspace;
// this variant needs none.
//
// How: it runs the generic pre path (split-K mixes kernel + finish/collapse
// kernel, unchanged) with its scratch -- the 256-byte status block and the
// split-K partial sums -- in the file-scope buffer below.  The buffer is part
// of the library image, so every GPU that loads the library holds its
// kNoallocScratchBytes until the process exits.  Its device address is looked
// up with cudaGetSymbolAddress once per device, on the first call made with
// that device current (and again if the device's context has been replaced,
// e.g. after cudaDeviceReset, which unloads the module and the buffer with it).
#include <mutex>

#include "hc_internal.cuh"

namespace hc {
namespace {

constexpr size_t kNoallocScratchBytes = (size_t)4 << 20;   // 4 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch on `device` (which must be current), cached
// per device under the id of the context it was looked up in.
void *scratch_address(int device, cudaError_t *err)
{
    static std::mutex mu;
    static void *addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    if (device < 0 || device >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = context_id();   // 0 before the runtime has made one current
    if (addr[device] == nullptr || ctx == 0 || ctx != ctx_of[device]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return nullptr;
        }
        addr[device] = p;
        ctx_of[device] = context_id();   // the look-up has made the device's context current
    }
    return addr[device];
}

}  // namespace
}  // namespace hc

extern "C" int hc_pre_fused_noalloc(const float *x, const float *fn_w, const float *scale,
                                    const float *base, int T, int s, int d, int iters, float eps,
                                    float *pre, float *post, float *comb, float *y, void *stream)
{
    if (hc_pre_workspace_bytes(T, s, d) == 0)   // 0: the shape is outside the limits
        return HC_ERR_DIM;
    // This entry point always runs the generic path: only its scratch (the status block
    // and the split-K partials) has to fit.
    const size_t need = hc::generic_workspace_bytes(T, s, d);
    if (need > hc::kNoallocScratchBytes)
        return HC_ERR_TOO_LARGE;
    if (T == 0)
        return HC_OK;
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess)
        return HC_ERR_CUDA;
    cudaError_t err = cudaSuccess;
    void *ws = hc::scratch_address(device, &err);
    if (ws == nullptr)
        return HC_ERR_CUDA;
    // Nothing in the buffer has to start at zero on this path: every partial sum
    // is written before it is read, and these kernels never touch the status block.
    return hc_pre_fused_path(x, fn_w, scale, base, T, s, d, iters, eps, pre, post, comb, y, ws,
                             hc::kNoallocScratchBytes, stream, HC_PATH_GENERIC);
}
