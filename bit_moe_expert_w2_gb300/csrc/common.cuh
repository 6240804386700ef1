// Shared device helpers and the internal launch interface of libmoe_w2.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe_w2.h"

namespace moe_w2 {

// ------------------------------------------------------------------ layouts
//
// Activation operands (x for gate_up, h for down) are stored in the "T16"
// layout along their K dimension: inside every group of 16 consecutive
// elements, stored position 4a+b holds natural element 4b+a (a 4x4 transpose).
// The code expansion below produces bf16 pairs (c_r, c_{r+4}) and
// (c_{r+8}, c_{r+12}) of a 16-code word; in T16 order those are adjacent, so a
// mma.sync B fragment is one 64-bit load and a UMMA smem row is written in
// storage order.
__host__ __device__ __forceinline__ int t16_pos(int n) { return (n & ~15) | ((n & 3) << 2) | ((n >> 2) & 3); }

// ------------------------------------------------------------------ status
__device__ __forceinline__ void flag_status(uint32_t* st, uint32_t bits)
{
    if (st != nullptr && bits != 0) atomicOr(st, bits);
}

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ldg_stream_u4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ldg_u4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg_u16(const void* p)
{
    unsigned short r;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// ------------------------------------------------------------------ code expansion
//
// UE8M0 byte s, code c = sign<<1 | mag: value (+-1 or +-4) * 2^(s-127).  As bf16
// the exponent field is s (magnitude 1) or s+2 (magnitude 4), the mantissa is 0:
//   high byte = sign<<7 | (s + 2*mag) >> 1,  low byte = ((s & 1) << 7).
// The low byte is the same for all four codes of a block.  lut holds the four
// high bytes (index = code), lo the low byte in all four bytes.  s outside
// [1,252] gives lut = lo = 0 (the block counts as zero).
struct ScaleLut {
    uint32_t lut, lo;
};
__device__ __forceinline__ ScaleLut make_lut(uint32_t s)
{
    ScaleLut r;
    uint32_t h = s >> 1;
    bool ok = (s - 1u) <= 251u;
    r.lut = ok ? (h * 0x01010101u + 0x81800100u) : 0u;
    r.lo = ok ? ((s & 1u) * 0x80808080u) : 0u;
    return r;
}

// Selector for bf16 pairs (c_r, c_{r+4}) in the low half and (c_{r+8}, c_{r+12})
// in the high half of a 16-code word w (code i in bits 2i..2i+1).  Byte-perm
// nibbles: 4 (any of 4..7) picks the low byte, the code picks its high byte.
template <int R>
__device__ __forceinline__ uint32_t code_selector(uint32_t w)
{
    uint32_t t = (R == 0) ? (w << 4) : (R == 1) ? (w << 2) : (R == 2) ? w : (w >> 2);
    return (t & 0x30303030u) | 0x04040404u;
}
__device__ __forceinline__ uint32_t expand_pair(const ScaleLut& l, uint32_t sel)
{
    return __byte_perm(l.lut, l.lo, sel);
}

// ------------------------------------------------------------------ mma.sync (decode)
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// ------------------------------------------------------------------ workspace
struct Workspace {
    int32_t* sorted;       // [P]
    int32_t* inv;          // [P]
    int32_t* offsets;      // [E+1]
    int32_t* active;       // [E] active experts ascending
    int32_t* active_count; // [1]
    int4* tiles;           // GEMM tiles (expert, first slot, pairs, 0)
    int32_t* tile_count;   // [1]
    uint16_t* xa;          // prefill: activation rows in expert order [P][H]; decode: x per token [T][H]; T16 layout
    int32_t* counters;     // decode: per 32-row block of y, CTAs done (last one runs the combine),
                           // then per tile, gate_up row blocks done (down items wait for their tile),
                           // then the decode item queue
    uint16_t* h;           // SiLU(gate)*up rows in expert order, T16 layout [P][I]
    float* stage;          // per-pair outputs times router weight, slot t*k+j [P][H]
    size_t bytes;
};

Workspace carve_workspace(void* base, int32_t T, int32_t k, int32_t E, int32_t H, int32_t I);
int64_t max_tiles(int64_t P, int32_t E, bool decode);

// ------------------------------------------------------------------ launches
// Optional profiling events recorded between phases (see moe_w2_forward_traced).
// During stream capture the events become external record nodes, so each graph
// replay records them and cudaEventElapsedTime works on replays.
struct PhaseEvents {
    cudaEvent_t e[4];
    cudaError_t record(int i, cudaStream_t s) const
    {
        if (!e[i]) return cudaSuccess;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        cudaError_t r = cudaStreamIsCapturing(s, &cs);
        if (r != cudaSuccess) return r;
        return cudaEventRecordWithFlags(e[i], s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
    }
};

cudaError_t launch_permute(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* sorted, int32_t* inv,
                           int32_t* offsets, int32_t* active, int32_t* active_count, int4* tiles,
                           int32_t* tile_count, int32_t tile_rows, const uint16_t* x, uint16_t* x_t16, int32_t H,
                           int32_t* counters, int32_t n_counters, uint16_t* y, uint32_t* status, cudaStream_t s);

cudaError_t launch_decode(const uint16_t* x, const int32_t* ids, const float* weights,
                          const moe_w2_planes& w, int32_t T, int32_t k, const Workspace& ws, uint16_t* y,
                          uint32_t* status, cudaStream_t s, const PhaseEvents& ev);

cudaError_t launch_prefill(const uint16_t* x, const int32_t* ids, const float* weights, const moe_w2_planes& w,
                           int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status,
                           cudaStream_t s, const PhaseEvents& ev);

cudaError_t launch_requant(const uint8_t* e2m1, const uint8_t* e4m3, const float* scale_2, int64_t n,
                           int64_t rows, int64_t K, uint8_t* codes, uint8_t* ue8m0, uint32_t* status,
                           cudaStream_t s);

int sm_count();

}  // namespace moe_w2
