// moe_w2_forward_noalloc: the layer forward with its scratch in a fixed device
// array that the library owns.
//
// Some callers cannot call cudaMalloc at the point where they run the layer:
// an allocator that must not grow, a process whose device memory is already
// handed out in full, or code that runs where an allocation would have to
// synchronise the device.  They cannot provide the workspace moe_w2_forward
// asks for, so this entry point takes its scratch from g_noalloc_workspace
// below instead.  The pages describe no such entry point.
//
// Set-up: the first call on each device, with that device current, looks up
// the array's device address with cudaGetSymbolAddress and keeps it; later
// calls on that device reuse it.  Make that first call before any stream
// capture starts.  The array is shared by every call on the device, so calls
// that may run at the same time (different streams or threads without an
// ordering between them) race on it: order them, for example on one stream.
// Nothing in it has to start at zero: the permute kernel zeroes the combine
// counters on every call and every other part is written before it is read.
#include <mutex>

#include <cuda_runtime.h>

#include "moe_w2.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_workspace[MOE_W2_NOALLOC_WORKSPACE_BYTES];

void* g_noalloc_ptr[kMaxDevices];
std::mutex g_noalloc_mu;

}  // namespace

extern "C" moe_w2_status moe_w2_forward_noalloc(const void* x_bf16, const int32_t* topk_ids,
                                                const float* topk_weights, const moe_w2_planes* w, int32_t T,
                                                int32_t top_k, void* y_bf16, uint32_t* dev_status, void* stream)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const size_t need = moe_w2_forward_workspace_size(T, top_k, w->num_experts, w->hidden, w->inter);
    if (need > MOE_W2_NOALLOC_WORKSPACE_BYTES) return MOE_W2_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_W2_ERR_CUDA;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return MOE_W2_ERR_CUDA;
            g_noalloc_ptr[dev] = p;
        }
        ws = g_noalloc_ptr[dev];
    }
    return moe_w2_forward(x_bf16, topk_ids, topk_weights, w, T, top_k, y_bf16, ws, MOE_W2_NOALLOC_WORKSPACE_BYTES,
                          dev_status, stream);
}
