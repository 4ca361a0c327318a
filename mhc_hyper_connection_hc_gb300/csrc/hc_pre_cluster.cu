// hc_pre_cluster.cu -- the fused single-launch pre-chain path (thread-block clusters).
#include "hc_internal.cuh"

namespace hc {

bool cluster_shape_ok(int, int) { return false; }
bool cluster_supported(int, int) { return false; }

cudaError_t launch_pre_cluster(const float *, const float *, const float *, const float *, int, int,
                               int, int, float, float *, float *, float *, float *, void *,
                               cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace hc
