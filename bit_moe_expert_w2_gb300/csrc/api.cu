// C ABI of libmoe_w2: host-side validation, workspace layout and launch order.
// The entry points only enqueue work on the caller's stream; nothing here
// allocates, frees or synchronises.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace moe_w2 {

namespace {

constexpr int32_t kPrefillTileRows = 256;   // pairs per prefill tile (tcgen05 N <= 256)
constexpr int32_t kDecodeTileRows = 4;      // pairs per decode tile (MMA N = 32: kActDigits rows per pair)
constexpr int32_t kDecodeMmaTileRows = 16;  // pairs per tile of the mma.sync decode kernel
constexpr int64_t kDecodeStreamMaxPairs = 16; // steps with at most this many pairs take the stream-K kernel
constexpr int64_t kDecodeMmaMaxPairs = 16;  // ... or, when it is deselected, the mma.sync kernel
constexpr int64_t kDecodeTargetItems = 1200; // down items per step that keep every CTA busy
constexpr int64_t kDecodeSplitMaxPairs = 32;  // steps of up to this many pairs may split gate_up K in two
constexpr int32_t kDecodeMinSegChunks = 2;   // at least 2 chunks of 256 K per decode item
constexpr int64_t kDecodeMaxSegments = 16;   // K segments per row block

int g_sm_count[kMaxDevices];
int g_cc_ok[kMaxDevices];   // 0 = unknown, 1 = ok, 2 = not sm_103
std::mutex g_mu;

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool layer_shape_ok(int32_t E, int32_t H, int32_t I)
{
    return E >= 1 && E <= MOE_W2_MAX_EXPERTS && H >= 256 && I >= 256 && H % 256 == 0 && I % 256 == 0 &&
           (int64_t)H * I <= ((int64_t)1 << 31);
}

}  // namespace

moe_w2_status check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_W2_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_cc_ok[dev] == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_W2_ERR_CUDA;
        g_sm_count[dev] = sms;
        g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return g_cc_ok[dev] == 1 ? MOE_W2_OK : MOE_W2_ERR_DEVICE;
}

std::atomic<int> g_force_timeout{0};
std::atomic<int> g_decode_stream{1};   // moe_w2_set_decode_stream

DepWait dependency_wait()
{
    if (g_force_timeout.load(std::memory_order_relaxed)) return DepWait{1, 200000ll};
    return DepWait{0, 4000000000ll};
}

std::mutex& init_mutex()
{
    static std::mutex mu;
    return mu;
}

int sm_count()
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int64_t max_tiles(int64_t P, int32_t E, bool decode)
{
    return P / (decode ? kDecodeTileRows : kPrefillTileRows) + E + 1;
}

DecodeSplit decode_split(int64_t P, int32_t E, int32_t H, int32_t I)
{
    // down: each 128-row block's K in s_dn equal segments, as many as keep a
    // small step's down phase in several short items per CTA
    DecodeSplit d{};
    const int64_t tiles = std::max<int64_t>(1, std::min<int64_t>(P, E));
    const int32_t nch_dn = I / 256;
    const int64_t rbd = H / 128;
    int64_t want = (kDecodeTargetItems + tiles * rbd - 1) / (tiles * rbd);
    want = std::min<int64_t>(want, std::max<int64_t>(1, 64 / std::max<int64_t>(1, P)));
    want = std::max<int64_t>(1, std::min<int64_t>({want, (int64_t)std::max(1, nch_dn / kDecodeMinSegChunks),
                                                    (int64_t)kDecodeMaxSegments}));
    d.l_dn = (int32_t)((nch_dn + want - 1) / want);
    d.s_dn = (nch_dn + d.l_dn - 1) / d.l_dn;
    return d;
}

// The block-scaled kernel loads weight-row scale groups by TMA, whose rows
// (H/32, I/32 bytes) must be multiples of 16 bytes.
bool decode_use_stream(int64_t P, int32_t H, int32_t I)
{
    // (its scale tiles hold whole scale rows of at most 224 bytes)
    return g_decode_stream.load(std::memory_order_relaxed) != 0 && P <= kDecodeStreamMaxPairs && H % 512 == 0 &&
           I % 512 == 0 && H <= 7168 && I <= 7168;
}

bool decode_use_mma(int64_t P, int32_t H, int32_t I)
{
    return P <= kDecodeMmaMaxPairs || H % 512 != 0 || I % 512 != 0;
}

int64_t decode_counter_count(int64_t P, int32_t E, int32_t H, int32_t I, bool mma)
{
    if (mma) return H / 32 + max_tiles(P, E, true) + 1;   // row blocks of y, tiles, queue
    // h publications and split-K arrivals per (tile, 64-row block), then the queue
    const int64_t mt = max_tiles(P, E, true);
    return 2 * mt * (I / 64) + 1;
}

Workspace carve_workspace(void* base, int32_t T, int32_t k, int32_t E, int32_t H, int32_t I, bool cached, bool w4)
{
    Workspace w{};
    const int64_t P = (int64_t)T * k;
    const bool decode = T <= MOE_W2_DECODE_MAX_TOKENS;
    char* p = static_cast<char*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char* r = p ? p + off : nullptr;
        off += align256(bytes);
        return r;
    };
    w.sorted = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
    w.inv = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
    w.offsets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
    w.active = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * E));
    w.active_count = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * 2));
    w.tile_count = w.active_count + 1;
    w.tiles = reinterpret_cast<int4*>(take(sizeof(int4) * max_tiles(P, E, decode)));
    if (decode && !w4 && decode_use_stream(P, H, I)) {
        w.counters = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * stream_counter_count(P, H, I)));
        w.xd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * T * (H / 2)));
        w.sxd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * T * (H / 32)));
        w.hd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * P * (I / 2)));
        w.shd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * P * (I / 32)));
        w.stage = reinterpret_cast<float*>(take(sizeof(float) * P * H));
        w.gu_part = reinterpret_cast<float*>(take(sizeof(float) * stream_part_floats()));
    } else if (decode && (w4 || decode_use_mma(P, H, I))) {
        w.counters = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * decode_counter_count(P, E, H, I, true)));
        w.xa = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * T * H));
        w.h = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * P * I));
        w.stage = reinterpret_cast<float*>(take(sizeof(float) * P * H));
    } else if (decode) {
        w.split = decode_split(P, E, H, I);
        w.counters = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * decode_counter_count(P, E, H, I, false)));
        w.xd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * T * (H / 2)));
        w.sxd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * T * (H / 32)));
        w.hd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * P * (I / 2)));
        w.shd = reinterpret_cast<uint8_t*>(take((size_t)kActDigits * P * (I / 32)));
        w.stage = reinterpret_cast<float*>(take(sizeof(float) * w.split.s_dn * P * H));
        if (P <= kDecodeSplitMaxPairs)
            w.gu_part = reinterpret_cast<float*>(take(sizeof(float) * 2 * P * 2 * I));
    } else {
        w.xa = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * P * H));
        w.h = reinterpret_cast<uint16_t*>(take(sizeof(uint16_t) * P * I));
        w.stage = reinterpret_cast<float*>(take(sizeof(float) * P * H));
    }
    if (cached) w.ids_eff = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
    w.bytes = off;
    return w;
}

// moe_w2_forward and its variants.  slot_of (nullable) is the residency table of
// an expert cache: routed id -> slot of w, negative when not resident.
moe_w2_status forward_impl(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                           const LayerPlanes* w, const int32_t* slot_of, int32_t n_route, int32_t T, int32_t top_k,
                           void* y_bf16, void* workspace, size_t workspace_bytes, uint32_t* misses,
                           uint32_t* dev_status, void* stream, void* const* phase_events)
{
    if (!w || T < 0 || top_k < 1 || top_k > MOE_W2_MAX_TOP_K) return MOE_W2_ERR_INVALID_ARG;
    if (w->num_experts < 1 || w->num_experts > MOE_W2_MAX_EXPERTS) return MOE_W2_ERR_INVALID_ARG;
    if (!layer_shape_ok(w->num_experts, w->hidden, w->inter)) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)T * top_k > MOE_W2_MAX_PAIRS) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_W2_OK;
    if (!x_bf16 || !topk_ids || !topk_weights || !y_bf16 || !workspace || !w->w13_codes || !w->w13_scales ||
        !w->w2_codes || !w->w2_scales || (w->w4 && (!w->w13_scale_2 || !w->w2_scale_2)))
        return MOE_W2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MOE_W2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x_bf16) & 15) != 0 || (reinterpret_cast<uintptr_t>(y_bf16) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(w->w13_codes) & 15) != 0 || (reinterpret_cast<uintptr_t>(w->w2_codes) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(w->w13_scales) & 15) != 0 || (reinterpret_cast<uintptr_t>(w->w2_scales) & 15) != 0)
        return MOE_W2_ERR_INVALID_ARG;
    if (w->w4 && ((reinterpret_cast<uintptr_t>(w->w13_scale_2) & 3) != 0 ||
                  (reinterpret_cast<uintptr_t>(w->w2_scale_2) & 3) != 0))
        return MOE_W2_ERR_INVALID_ARG;
    const int32_t E = w->num_experts, H = w->hidden, I = w->inter;
    const bool cached = slot_of != nullptr;
    Workspace ws = carve_workspace(workspace, T, top_k, E, H, I, cached, w->w4);
    if (workspace_bytes < ws.bytes) return MOE_W2_ERR_WORKSPACE;
    moe_w2_status st = check_device();
    if (st != MOE_W2_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool decode = T <= MOE_W2_DECODE_MAX_TOKENS;
    const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
    uint16_t* y = static_cast<uint16_t*>(y_bf16);
    PhaseEvents ev{};
    for (int i = 0; i < 4; ++i) ev.e[i] = phase_events ? static_cast<cudaEvent_t>(phase_events[i]) : nullptr;
    if (ev.record(0, s) != cudaSuccess) return MOE_W2_ERR_CUDA;
    const int64_t P = (int64_t)T * top_k;
    // the FP4 layer's decode steps all take the mma.sync kernel
    const bool use_stream = decode && !w->w4 && decode_use_stream(P, H, I);
    const bool mma = decode && !use_stream && (w->w4 || decode_use_mma(P, H, I));
    const bool digits = decode && !mma;   // x as e2m1 digit rows for a block-scaled kernel
    PermuteSlots slots{};
    if (cached) slots = PermuteSlots{slot_of, n_route, ws.ids_eff, misses};
    cudaError_t e = launch_permute(topk_ids, slots, T, top_k, E, ws.sorted, ws.inv, ws.offsets, ws.active,
                                   ws.active_count, ws.tiles, ws.tile_count,
                                   !decode ? kPrefillTileRows : mma ? kDecodeMmaTileRows : kDecodeTileRows,
                                   decode ? x : nullptr, mma ? ws.xa : nullptr, digits ? ws.xd : nullptr,
                                   digits ? ws.sxd : nullptr, H, ws.counters,
                                   !decode ? 0
                                   : use_stream ? (int32_t)stream_counter_count(P, H, I)
                                            : (int32_t)decode_counter_count(P, E, H, I, mma),
                                   decode ? y : nullptr,
                                   dev_status, s);
    if (e != cudaSuccess) return MOE_W2_ERR_CUDA;
    // the later kernels read the ids only to tell kept pairs from left-out ones
    const int32_t* ids = cached ? ws.ids_eff : topk_ids;
    const moe_w2_planes p2{w->w13_codes, w->w13_scales, w->w2_codes, w->w2_scales, E, H, I};
    if (use_stream) {
        e = launch_decode_stream(ids, topk_ids, slot_of, n_route, topk_weights, p2, T, top_k, ws, y, dev_status, s,
                                 ev);
    } else if (mma) {
        e = launch_decode_mma(ids, topk_weights, *w, T, top_k, ws, y, dev_status, s, ev);
    } else if (decode) {
        e = launch_decode(x, ids, topk_weights, p2, T, top_k, ws, y, dev_status, s, ev);
    } else {
        e = launch_prefill(x, ids, topk_weights, *w, T, top_k, ws, y, dev_status, s, ev);
    }
    if (e != cudaSuccess) return MOE_W2_ERR_CUDA;
    return ev.record(3, s) == cudaSuccess ? MOE_W2_OK : MOE_W2_ERR_CUDA;
}

LayerPlanes planes_of(const moe_w2_planes* w)
{
    if (!w) return LayerPlanes{};
    return LayerPlanes{false, w->w13_codes, w->w13_scales, w->w2_codes, w->w2_scales, nullptr, nullptr,
                       w->num_experts, w->hidden, w->inter};
}

LayerPlanes planes_of(const moe_w4_planes* w)
{
    if (!w) return LayerPlanes{};
    return LayerPlanes{true, w->w13_e2m1, w->w13_e4m3, w->w2_e2m1, w->w2_e4m3, w->w13_scale_2, w->w2_scale_2,
                       w->num_experts, w->hidden, w->inter};
}

}  // namespace moe_w2

using namespace moe_w2;

extern "C" {

int moe_w2_version(void) { return (0 << 16) | 1; }

moe_w2_status moe_w2_debug_force_pipeline_timeout(int32_t enable)
{
    g_force_timeout.store(enable != 0 ? 1 : 0, std::memory_order_relaxed);
    return MOE_W2_OK;
}

moe_w2_status moe_w2_set_decode_stream(int32_t enable)
{
    g_decode_stream.store(enable != 0 ? 1 : 0, std::memory_order_relaxed);
    return MOE_W2_OK;
}

const char* moe_w2_status_string(moe_w2_status s)
{
    switch (s) {
        case MOE_W2_OK: return "ok";
        case MOE_W2_ERR_INVALID_ARG: return "invalid argument";
        case MOE_W2_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_W2_ERR_WORKSPACE: return "workspace too small";
        case MOE_W2_ERR_CUDA: return "CUDA error";
        case MOE_W2_ERR_DEVICE: return "device is not compute capability 10.3";
    }
    return "unknown status";
}

size_t moe_w2_forward_workspace_size(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I)
{
    if (T < 0 || top_k < 1 || top_k > MOE_W2_MAX_TOP_K || !layer_shape_ok(E, H, I)) return 0;
    if ((int64_t)T * top_k > MOE_W2_MAX_PAIRS) return 0;
    return carve_workspace(nullptr, T, top_k, E, H, I).bytes;
}

int moe_w2_forward_path(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I)
{
    if (T <= 0 || moe_w2_forward_workspace_size(T, top_k, E, H, I) == 0) return MOE_W2_PATH_NONE;
    if (T > MOE_W2_DECODE_MAX_TOKENS) return MOE_W2_PATH_PREFILL;
    const int64_t P = (int64_t)T * top_k;
    if (decode_use_stream(P, H, I)) return MOE_W2_PATH_DECODE_STREAM;
    return decode_use_mma(P, H, I) ? MOE_W2_PATH_DECODE_MMA : MOE_W2_PATH_DECODE_BLOCK_SCALED;
}

moe_w2_status moe_w2_permute(const int32_t* topk_ids, int32_t T, int32_t top_k, int32_t E, int32_t* sorted_pairs,
                             int32_t* inv_pairs, int32_t* expert_offsets, uint32_t* dev_status, void* stream)
{
    if (T < 0 || top_k < 1 || top_k > MOE_W2_MAX_TOP_K || E < 1 || E > MOE_W2_MAX_EXPERTS)
        return MOE_W2_ERR_INVALID_ARG;
    if ((int64_t)T * top_k > MOE_W2_MAX_PAIRS) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets || (T > 0 && (!topk_ids || !sorted_pairs || !inv_pairs))) return MOE_W2_ERR_INVALID_ARG;
    moe_w2_status st = check_device();
    if (st != MOE_W2_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_permute(topk_ids, PermuteSlots{}, T, top_k, E, sorted_pairs, inv_pairs, expert_offsets,
                                   nullptr, nullptr,
                                   nullptr, nullptr, 1, nullptr, nullptr, nullptr, nullptr, 0, nullptr, 0, nullptr,
                                   dev_status, s);
    return e == cudaSuccess ? MOE_W2_OK : MOE_W2_ERR_CUDA;
}

moe_w2_status moe_w2_forward_traced(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                                    const moe_w2_planes* w, int32_t T, int32_t top_k, void* y_bf16,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_status, void* stream,
                                    void* const* phase_events)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const LayerPlanes p = planes_of(w);
    return forward_impl(x_bf16, topk_ids, topk_weights, &p, nullptr, 0, T, top_k, y_bf16, workspace, workspace_bytes,
                        nullptr, dev_status, stream, phase_events);
}

moe_w2_status moe_w2_forward(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                             const moe_w2_planes* w, int32_t T, int32_t top_k, void* y_bf16, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_status, void* stream)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const LayerPlanes p = planes_of(w);
    return forward_impl(x_bf16, topk_ids, topk_weights, &p, nullptr, 0, T, top_k, y_bf16, workspace, workspace_bytes,
                        nullptr, dev_status, stream, nullptr);
}

moe_w2_status moe_w4_forward_traced(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                                    const moe_w4_planes* w, int32_t T, int32_t top_k, void* y_bf16,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_status, void* stream,
                                    void* const* phase_events)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const LayerPlanes p = planes_of(w);
    return forward_impl(x_bf16, topk_ids, topk_weights, &p, nullptr, 0, T, top_k, y_bf16, workspace, workspace_bytes,
                        nullptr, dev_status, stream, phase_events);
}

size_t moe_w4_forward_workspace_size(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I)
{
    if (moe_w2_forward_workspace_size(T, top_k, E, H, I) == 0) return 0;
    return carve_workspace(nullptr, T, top_k, E, H, I, false, true).bytes;
}

moe_w2_status moe_w4_forward(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                             const moe_w4_planes* w, int32_t T, int32_t top_k, void* y_bf16, void* workspace,
                             size_t workspace_bytes, uint32_t* dev_status, void* stream)
{
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const LayerPlanes p = planes_of(w);
    return forward_impl(x_bf16, topk_ids, topk_weights, &p, nullptr, 0, T, top_k, y_bf16, workspace, workspace_bytes,
                        nullptr, dev_status, stream, nullptr);
}

size_t moe_w2_forward_cached_workspace_size(int32_t T, int32_t top_k, int32_t num_slots, int32_t H, int32_t I)
{
    if (moe_w2_forward_workspace_size(T, top_k, num_slots, H, I) == 0) return 0;
    return carve_workspace(nullptr, T, top_k, num_slots, H, I, true).bytes;
}

moe_w2_status moe_w2_forward_cached(const void* x_bf16, const int32_t* topk_ids, const float* topk_weights,
                                    const moe_w2_planes* w, const int32_t* slot_of_expert,
                                    int32_t num_routed_experts, int32_t T, int32_t top_k, void* y_bf16,
                                    void* workspace, size_t workspace_bytes, uint32_t* miss_counter,
                                    uint32_t* dev_status, void* stream)
{
    if (num_routed_experts < 1 || num_routed_experts > MOE_W2_MAX_ROUTED_EXPERTS) return MOE_W2_ERR_INVALID_ARG;
    if (T > 0 && !slot_of_expert) return MOE_W2_ERR_INVALID_ARG;
    if (!w) return MOE_W2_ERR_INVALID_ARG;
    const LayerPlanes p = planes_of(w);
    return forward_impl(x_bf16, topk_ids, topk_weights, &p, slot_of_expert, num_routed_experts, T, top_k, y_bf16,
                        workspace, workspace_bytes, miss_counter, dev_status, stream, nullptr);
}

moe_w2_status moe_w2_requant(const uint8_t* e2m1, const uint8_t* e4m3, const float* scale_2, int64_t n,
                             int64_t rows, int64_t K, uint8_t* codes, uint8_t* ue8m0, uint32_t* dev_status,
                             void* stream)
{
    return moe_w2_requant_ex(e2m1, e4m3, scale_2, n, rows, K, 0u, codes, ue8m0, dev_status, stream);
}

moe_w2_status moe_w2_requant_ex(const uint8_t* e2m1, const uint8_t* e4m3, const float* scale_2, int64_t n,
                                int64_t rows, int64_t K, uint32_t options, uint8_t* codes, uint8_t* ue8m0,
                                uint32_t* dev_status, void* stream)
{
    if ((options & ~MOE_W2_REQUANT_BALANCE_ZERO_SIGNS) != 0u) return MOE_W2_ERR_INVALID_ARG;
    if (n < 0 || rows < 0 || K < 0) return MOE_W2_ERR_INVALID_ARG;
    if (K % 32 != 0) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (n == 0 || rows == 0 || K == 0) return MOE_W2_OK;
    if (rows > ((int64_t)1 << 40) / K || n > ((int64_t)1 << 50) / (rows * K)) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (!e2m1 || !e4m3 || !scale_2 || !codes || !ue8m0) return MOE_W2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(e2m1) & 15) != 0 || (reinterpret_cast<uintptr_t>(e4m3) & 1) != 0 ||
        (reinterpret_cast<uintptr_t>(codes) & 7) != 0 || (reinterpret_cast<uintptr_t>(scale_2) & 3) != 0)
        return MOE_W2_ERR_INVALID_ARG;
    moe_w2_status st = check_device();
    if (st != MOE_W2_OK) return st;
    cudaError_t e = launch_requant(e2m1, e4m3, scale_2, n, rows, K, options, codes, ue8m0, dev_status,
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_W2_OK : MOE_W2_ERR_CUDA;
}

moe_w2_status moe_w2_requant_mxfp4(const uint8_t* e2m1, const uint8_t* scales, int64_t n, int64_t rows, int64_t K,
                                   uint32_t options, uint8_t* codes, uint8_t* ue8m0, uint32_t* dev_status,
                                   void* stream)
{
    if (n < 0 || rows < 0 || K < 0) return MOE_W2_ERR_INVALID_ARG;
    if ((options & ~MOE_W2_REQUANT_BALANCE_ZERO_SIGNS) != 0u) return MOE_W2_ERR_INVALID_ARG;
    if (K % 32 != 0) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (n == 0 || rows == 0 || K == 0) return MOE_W2_OK;
    if (rows > ((int64_t)1 << 40) / K || n > ((int64_t)1 << 50) / (rows * K)) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (!e2m1 || !scales || !codes || !ue8m0) return MOE_W2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(e2m1) & 15) != 0 || (reinterpret_cast<uintptr_t>(codes) & 7) != 0)
        return MOE_W2_ERR_INVALID_ARG;
    moe_w2_status st = check_device();
    if (st != MOE_W2_OK) return st;
    cudaError_t e = launch_requant_mxfp4(e2m1, scales, n, rows, K, options, codes, ue8m0, dev_status,
                                         static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_W2_OK : MOE_W2_ERR_CUDA;
}

moe_w2_status moe_w2_requant_fp8(const uint8_t* w8, const float* scales, int64_t n, int64_t rows, int64_t K,
                                 uint8_t* codes, uint8_t* ue8m0, uint32_t* dev_status, void* stream)
{
    if (n < 0 || rows < 0 || K < 0) return MOE_W2_ERR_INVALID_ARG;
    if (K % 32 != 0) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (n == 0 || rows == 0 || K == 0) return MOE_W2_OK;
    if (rows > ((int64_t)1 << 40) / K || n > ((int64_t)1 << 50) / (rows * K)) return MOE_W2_ERR_UNSUPPORTED_SHAPE;
    if (!w8 || !scales || !codes || !ue8m0) return MOE_W2_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w8) & 15) != 0 || (reinterpret_cast<uintptr_t>(codes) & 7) != 0 ||
        (reinterpret_cast<uintptr_t>(scales) & 3) != 0)
        return MOE_W2_ERR_INVALID_ARG;
    moe_w2_status st = check_device();
    if (st != MOE_W2_OK) return st;
    cudaError_t e = launch_requant_fp8(w8, scales, n, rows, K, codes, ue8m0, dev_status,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_W2_OK : MOE_W2_ERR_CUDA;
}

}  // extern "C"
