// Blackwell (sm_103a) primitives in inline PTX: mbarriers with bounded waits,
// TMA tensor loads, tcgen05 (tensor memory alloc, UMMA issue/commit, loads) and
// the shared-memory matrix descriptor for the 128-byte-swizzled K-major layout.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "common.cuh"

namespace moe_w2 {

// Bit OR-ed into the device status when a pipeline wait gives up (a bug, never
// expected): the kernel stops its work loop, releases tensor memory and returns.
constexpr uint32_t kDevPipelineTimeout = MOE_W2_DEV_PIPELINE_TIMEOUT;
constexpr long long kWaitLimitCycles = 4000000000ll;   // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// The same with relaxed memory semantics: for an arrival that only announces
// the bytes a TMA copy will complete, with no earlier write of this thread to
// publish (a release arrival would first wait for every outstanding memory
// operation of the thread, such as a slow atomic).
__device__ __forceinline__ void mbar_arrive_expect_tx_relaxed(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false if `abort` was raised elsewhere or the limit passed (then
// this thread raises `abort`).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            return false;
        }
    }
}

// CTA-wide barrier that counts threads, for the end of a kernel whose warps ran
// roles on single lanes: __syncthreads (bar.sync) counts a warp at each of its
// arrivals and its lanes may arrive apart after diverging, so it could release
// before every warp is done; the non-aligned barrier.sync waits for all threads.
__device__ __forceinline__ void cta_barrier_all_threads() { asm volatile("barrier.sync 0;" ::: "memory"); }

// Bounded wait as mbar_wait for a thread off the critical path: it sleeps about
// `ns` between polls, so that a warp that waits leaves its sub-partition's issue
// slots to the warps that work.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort = 1;
            return false;
        }
    }
}

// The whole warp waits (bounded) while lane 0 alone polls, sleeping about `ns`
// between polls; every lane gets lane 0's result, and the lanes' later accesses
// are ordered after lane 0's observation of the phase (__syncwarp).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort, uint32_t ns)
{
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_sleep(bar, parity, abort, ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Both barriers' phases complete (bounded as mbar_wait); the two first polls are
// issued back to back so that their latencies overlap.
__device__ __forceinline__ bool mbar_wait2(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, volatile int* abort)
{
    const bool r1 = mbar_try_wait(b1, p1), r2 = mbar_try_wait(b2, p2);
    if (r1 && r2) return true;
    return (r1 || mbar_wait(b1, p1, abort)) && (r2 || mbar_wait(b2, p2, abort));
}

// ------------------------------------------------------------------ shared-memory access
// Explicit shared-space loads/stores for tiles handed over through mbarriers:
// they stay ordered with the barrier operations around them (a generic-address
// access to a TMA-filled tile was observed to be reordered past the release).
__device__ __forceinline__ uint4 lds_u4(uint32_t saddr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(saddr)
                 : "memory");
    return r;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t saddr)
{
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(saddr) : "memory");
    return r;
}
__device__ __forceinline__ void sts_u4(uint32_t saddr, const uint4& v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t c0, int32_t c1, int32_t c2,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}
// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16); no
// completion to wait for.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on an mbarrier when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes.  The load and its
// wait are one asm statement: tcgen05.ld writes the destination registers
// asynchronously, so nothing may touch them before tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, no negation or sparsity; N in bits 17..22 (N >> 3), M in 24..28 (M >> 4).
__host__ __device__ __forceinline__ uint32_t idesc_bf16_f32(uint32_t M, uint32_t N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Shared-memory descriptor of a K-major operand stored in the 128-byte swizzle
// layout: rows of 128 bytes (64 bf16), 8-row groups 1024 bytes apart (stride
// byte offset), 16-byte chunk j of row r at position j ^ (r % 8).  The tile base
// must be 1024-byte aligned; moving along K inside the 128-byte row is done by
// advancing the start address (32 bytes per K = 16 step).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Byte offset of 16-byte chunk j (0..7) of row r in a 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t j)
{
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((j ^ (r & 7u)) << 4);
}

// ------------------------------------------------------------------ block-scaled MMA (decode)
//
// tcgen05.mma kind::mxf4 (A and B packed e2m1, two per byte) with UE8M0 block
// scales, one per 32 K per row of A and per row of B (scale_vec::2X: an MMA of K
// = 64 takes two consecutive scale bytes), A read from tensor memory.  Layouts
// measured on GB300 with in-bounds probes of the instruction (M = 128, N = 16):
//  - A: lane m holds row m; column j, nibble i (bits 4i..4i+3) holds K index
//    8j + i, so one MMA reads 8 columns.
//  - B (shared memory, K-major, 128B-swizzled rows): nibble h (low first) of
//    byte b holds K index 2b + h; one MMA reads 32 bytes of each row.
//  - A scales: the scale word of row m is read from lane m of the column
//    (scale_A_tmem + m / 32); bytes sf_id and sf_id + 1 (sf_id 0 or 2) scale K
//    0..31 and 32..63 of the MMA.  So the warp owning lanes 32w..32w+31 writes
//    its rows' scale words into column scale_A_tmem + w.
//  - B scales: the scale word of B row n is read from lane n % 32 of column
//    scale_B_tmem in the lane quadrant of the output row, same byte use, so
//    every quadrant holds a copy.
//  - Scale-factor columns start on a 4-column boundary (an odd column raised a
//    misaligned-address fault).
// Instruction descriptor (block-scaled form): b_sf_id bits 4-5, A/B format bits
// 7-9 / 10-12 (1 = e2m1 for kind::mxf4), N >> 3 in bits 17-22, scale format bit
// 23 (1 = UE8M0), M >> 4 in bits 24-28, a_sf_id bits 29-30; K-major A and B,
// dense, fp32 D.
__host__ __device__ __forceinline__ uint32_t idesc_mxf4(uint32_t M, uint32_t N, uint32_t a_sf, uint32_t b_sf)
{
    return (b_sf << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) | (a_sf << 29);
}
__device__ __forceinline__ void umma_mxf4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n}\n"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// 32 columns of A, two columns of A scale words and two of B scale words from
// this warp's registers into its TMEM lane quadrant, completed before returning
// (the registers are read until tcgen05.wait::st, so store and wait share one asm).
__device__ __forceinline__ void tmem_st_stage4(uint32_t ta, const uint32_t (&r)[32], uint32_t tsa0, uint32_t sa0,
                                               uint32_t tsa1, uint32_t sa1, uint32_t tsb0, uint32_t sb0, uint32_t tsb1,
                                               uint32_t sb1)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%33], {%34};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%35], {%36};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%37], {%38};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%39], {%40};\n"
        "tcgen05.wait::st.sync.aligned;" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(tsa0), "r"(sa0), "r"(tsa1), "r"(sa1),
        "r"(tsb0), "r"(sb0), "r"(tsb1), "r"(sb1)
        : "memory");
}

// tmem_st_stage4 in two halves: the A stage and its two scale words now (not
// waited for), the B scale words later, when they have come, and then the wait
// for all six stores.  The registers of the first half are read until the
// wait, so the second asm takes them as inputs too (they stay untouched).
__device__ __forceinline__ void tmem_st_a_sfa(uint32_t ta, const uint32_t (&r)[32], uint32_t tsa0, uint32_t sa0,
                                              uint32_t tsa1, uint32_t sa1)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%33], {%34};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%35], {%36};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(tsa0), "r"(sa0), "r"(tsa1), "r"(sa1)
        : "memory");
}
__device__ __forceinline__ void tmem_st_sfb_wait(const uint32_t (&r)[32], uint32_t sa0, uint32_t sa1, uint32_t tsb0,
                                                 uint32_t sb0, uint32_t tsb1, uint32_t sb1)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%32], {%33};\n"
        "tcgen05.st.sync.aligned.32x32b.x1.b32 [%34], {%35};\n"
        "tcgen05.wait::st.sync.aligned;" ::"r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(tsb0), "r"(sb0), "r"(tsb1), "r"(sb1), "r"(sa0), "r"(sa1)
        : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes (load and wait in one asm).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ non-bulk async copies
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
// The barrier gets one arrival once all of this thread's earlier cp.async copies
// have landed (its expected count includes that arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// ------------------------------------------------------------------ host side (route.cu)
// 2-D tensor map [rows][cols] (row-major) of bf16 or uint8, box {box_cols, box_rows}.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t cols,
                         uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);
// 3-D tensor map of uint8 [planes][rows][cols] (row-major, planes contiguous),
// box {box_cols, box_rows, box_planes}: e.g. the gate and up halves of an
// expert's w13 plane as two consecutive planes of I rows.
cudaError_t make_tmap_3d_u8(CUtensorMap* map, const void* base, int64_t planes, int64_t rows, int64_t cols,
                            uint32_t box_cols, uint32_t box_rows, uint32_t box_planes, int swizzle_bytes);
// Tensor map of uint8 elements of any rank (1-5): dims[0] contiguous, strides
// (bytes, multiples of 16) of dims 1.. in any order, e.g. the digit rows of an
// activation seen as {128 bytes of a chunk, row, chunk} with the chunk stride
// (128) below the row stride, so that a box lands chunk-major.
cudaError_t make_tmap_u8(CUtensorMap* map, const void* base, int rank, const int64_t* dims, const int64_t* strides,
                         const uint32_t* box, int swizzle_bytes);
cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted, const int32_t* offsets, int32_t E, int32_t k,
                          int32_t H, int64_t P, uint16_t* xs, cudaStream_t s);
cudaError_t launch_combine(const float* stage, const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t H,
                           int32_t n_seg, int64_t seg_stride, bool programmatic, uint16_t* y, cudaStream_t s);

}  // namespace moe_w2
