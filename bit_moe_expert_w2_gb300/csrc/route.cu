// Routing data movement shared by the decode and prefill paths, and the TMA
// tensor-map encoder.
//
// vLLM-Moet, page "The v0.24.0 port", section "Our hooks", "Deterministic
// unpermute" bullet: every pair's output row goes to its own slot
// (slot = token*top_k + j, a bijection) and each token's k slots are summed in a
// fixed order, so repeated runs are bit-identical.
//   gather   xs[q] = T16(x[sorted[q] / k]): activation rows in expert order, in
//            the T16 layout the GEMM kernels read (TMA-friendly contiguous rows
//            per expert)
//   combine  y[t] = bf16(sum_{j=0..k-1} stage[t*k + j]) over valid pairs, j in order
//            (decode: per slot also over the K segments of down, in order)
#include <algorithm>
#include <mutex>

#include "tc.cuh"

namespace moe_w2 {

namespace {

__global__ void gather_t16_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ sorted,
                                  const int32_t* __restrict__ offsets, int32_t E, int32_t k, int32_t H,
                                  uint16_t* __restrict__ xs)
{
    const int64_t groups = (int64_t)offsets[E] * (H / 16);
    const int gpr = H / 16;
    for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < groups;
         gi += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = gi / gpr;
        const int gcol = (int)(gi % gpr);
        const uint16_t* src = x + (int64_t)(sorted[q] / k) * H + gcol * 16;
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(src + 8));
        // natural words a.x=(x0,x1) a.y=(x2,x3) a.z=(x4,x5) a.w=(x6,x7) b.x=(x8,x9) ...
        uint4 o, t;
        o.x = __byte_perm(a.x, a.z, 0x5410);   // (x0, x4)
        o.y = __byte_perm(b.x, b.z, 0x5410);   // (x8, x12)
        o.z = __byte_perm(a.x, a.z, 0x7632);   // (x1, x5)
        o.w = __byte_perm(b.x, b.z, 0x7632);   // (x9, x13)
        t.x = __byte_perm(a.y, a.w, 0x5410);   // (x2, x6)
        t.y = __byte_perm(b.y, b.w, 0x5410);   // (x10, x14)
        t.z = __byte_perm(a.y, a.w, 0x7632);   // (x3, x7)
        t.w = __byte_perm(b.y, b.w, 0x7632);   // (x11, x15)
        uint16_t* dst = xs + q * H + gcol * 16;
        *reinterpret_cast<uint4*>(dst) = o;
        *reinterpret_cast<uint4*>(dst + 8) = t;
    }
}

// y[t] = bf16(sum over valid j, then over K segments, of stage[seg][t*k + j]).
// Launched as a programmatic dependent of the kernel that writes stage: it waits
// for that grid before reading (a no-op for an ordinary launch).
__global__ void combine_kernel(const float* __restrict__ stage, const int32_t* __restrict__ ids, int32_t T,
                               int32_t k, int32_t E, int32_t H, int32_t n_seg, int64_t seg_stride,
                               uint16_t* __restrict__ y)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // one thread per 4 consecutive outputs of a token; its k * n_seg slots are
    // loaded in batches of 8 (all loads of a batch in flight together) and
    // summed in (j, segment) order
    const int per_row = H / 4;
    const int nks = k * n_seg;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (int64_t)T * per_row;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_row;
        const int m = (int)(i % per_row) * 4;
        uint32_t valid = 0;   // bit j: slot j has an expert (k <= 16)
        for (int j = 0; j < k; ++j) valid |= (uint32_t)((unsigned)__ldg(ids + t * k + j) < (unsigned)E) << j;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int x0 = 0; x0 < nks; x0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int x = x0 + u, j = x / n_seg, sg = x - j * n_seg;
                v[u] = (x < nks && ((valid >> j) & 1u))
                           ? __ldcg(reinterpret_cast<const float4*>(stage + sg * seg_stride + (t * k + j) * H + m))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                acc.x += v[u].x;
                acc.y += v[u].y;
                acc.z += v[u].z;
                acc.w += v[u].w;
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(y + t * H + m) = o;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t get_encoder()
{
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (g_encode) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

}  // namespace

cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t cols, uint32_t box_cols,
                         uint32_t box_rows, int swizzle_bytes)
{
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    const int esz = bf16 ? 2 : 1;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_3d_u8(CUtensorMap* map, const void* base, int64_t planes, int64_t rows, int64_t cols,
                            uint32_t box_cols, uint32_t box_rows, uint32_t box_planes, int swizzle_bytes)
{
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)planes};
    cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(rows * cols)};
    cuuint32_t box[3] = {box_cols, box_rows, box_planes};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_u8(CUtensorMap* map, const void* base, int rank, const int64_t* dims, const int64_t* strides,
                         const uint32_t* box, int swizzle_bytes)
{
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = (cuuint64_t)dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i > 0) st[i - 1] = (cuuint64_t)strides[i - 1];
    }
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted, const int32_t* offsets, int32_t E, int32_t k,
                          int32_t H, int64_t P, uint16_t* xs, cudaStream_t s)
{
    const int64_t groups = P * (H / 16);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((groups + 255) / 256, (int64_t)sm_count() * 8));
    gather_t16_kernel<<<grid, 256, 0, s>>>(x, sorted, offsets, E, k, H, xs);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* stage, const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t H,
                           int32_t n_seg, int64_t seg_stride, bool programmatic, uint16_t* y, cudaStream_t s)
{
    const int64_t threads = (int64_t)T * (H / 4);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((threads + 255) / 256, (int64_t)sm_count() * 8));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel, stage, ids, T, k, E, H, n_seg, seg_stride, y);
}

}  // namespace moe_w2
