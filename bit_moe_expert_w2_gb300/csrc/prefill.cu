// Prefill path placeholder (tcgen05 kernels land next).
#include "common.cuh"

namespace moe_w2 {

cudaError_t launch_prefill(const uint16_t*, const int32_t*, const float*, const moe_w2_planes&, int32_t, int32_t,
                           const Workspace&, uint16_t*, uint32_t*, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace moe_w2
