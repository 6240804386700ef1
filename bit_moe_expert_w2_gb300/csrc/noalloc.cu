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
// Set-up: the first call in each CUDA context (normally a device's primary
// context), with that device current, checks the device and looks up the
// array's device address with cudaGetSymbolAddress; later calls in the same
// context reuse it.  A context is recognised by its ID, which CUDA never gives
// to another context in the process, so after cudaDeviceReset (which destroys
// the primary context and with it the array) the next call looks the address
// up again.  Make the first call before any stream capture starts.  The array
// is shared by every call in the context, so calls that may run at the same
// time (different streams or threads without an ordering between them) race on
// it: order them, for example on one stream.  Nothing in it has to start at
// zero: the permute kernel zeroes the combine counters on every call and every
// other part is written before it is read.
#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace {

constexpr int kSlots = 64;   // devices

static __device__ __align__(256) unsigned char g_noalloc_workspace[MOE_W2_NOALLOC_WORKSPACE_BYTES];

struct Cached {
    unsigned long long ctx_id;   // context the address belongs to (0 = none yet)
    void* ptr;
};
Cached g_noalloc[kSlots];
std::mutex g_noalloc_mu;

using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);

// ID of the current context, 0 when there is none (or it cannot be read).
unsigned long long current_ctx_id()
{
    static PfnCtxGetCurrent get_current = nullptr;
    static PfnCtxGetId get_id = nullptr;
    if (!get_current || !get_id) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
            return 0;
        get_current = reinterpret_cast<PfnCtxGetCurrent>(f1);
        get_id = reinterpret_cast<PfnCtxGetId>(f2);
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace

extern "C" moe_w2_status moe_w2_forward_noalloc(const void* x_bf16, const int32_t* topk_ids,
                                                const float* topk_weights, const moe_w2_planes* w, int32_t T,
                                                int32_t top_k, void* y_bf16, uint32_t* dev_status, void* stream)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const size_t need = moe_w2_forward_workspace_size(T, top_k, w->num_experts, w->hidden, w->inter);
    if (need > MOE_W2_NOALLOC_WORKSPACE_BYTES) return MOE_W2_ERR_WORKSPACE;
    // the device check comes first: on a device without an sm_103 image the
    // symbol lookup below would fail with a CUDA error
    const moe_w2_status dst = moe_w2::check_device();
    if (dst != MOE_W2_OK) return dst;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSlots) return MOE_W2_ERR_CUDA;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        Cached& c = g_noalloc[dev];
        const unsigned long long id = current_ctx_id();
        if (id == 0 || c.ctx_id != id || !c.ptr) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || !p) return MOE_W2_ERR_CUDA;
            // the lookup makes a context current if there was none: key on that one
            c.ctx_id = id != 0 ? id : current_ctx_id();
            c.ptr = p;
        }
        ws = c.ptr;
    }
    return moe_w2_forward(x_bf16, topk_ids, topk_weights, w, T, top_k, y_bf16, ws, MOE_W2_NOALLOC_WORKSPACE_BYTES,
                          dev_status, stream);
}
