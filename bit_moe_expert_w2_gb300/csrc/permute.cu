// Routing permutation: stable counting sort of pairs p = t*k + j by expert id.
//
// vLLM-Moet, page "The v0.24.0 port", section "Our hooks", deterministic
// unpermute bullet: valid sorted ids are a permutation of token*top_k+j, which
// lets the combine be a bijective placement plus a fixed-order sum.
//
// One CTA of 1024 threads does the whole permutation: warp w owns a contiguous
// slice of pairs; pass 1 counts per (warp, expert) in shared memory, a scan turns
// the counts into per-(warp, expert) write cursors, pass 2 walks each slice in
// order and writes every pair at its cursor (ranks within a 32-pair step come
// from match_any), so the result is the stable order without any sort network.
// The same launch also emits the active-expert list (decode scheduling) and the
// GEMM tile list (expert, first slot, pairs) with at most tile_rows pairs per
// tile.  Extra CTAs of the launch write x as the decode kernels read it: in T16
// order (mma.sync kernel) or as rows of packed e2m1 digits with UE8M0 bytes per
// 32 elements (block-scaled kernel, kActDigits rows per token).
//
// Behind an expert cache (page "vLLM-Moet wiki", BASE-cache paragraph; page "The
// v0.24.0 port", section "Our hooks", BASE-cache bullet) the planes hold E
// resident slots and a table maps each routed expert id to its slot, or to a
// negative value when the expert is not resident.  The permutation then sorts
// by slot; a pair whose expert is missing is left out like an invalid id (it
// contributes zero) but raises no status bit: it adds one to the caller's miss
// counter instead.  The slot of every pair (-1 when left out) goes to ids_eff,
// which the later kernels read in place of the routed ids.
#include <algorithm>

#include "common.cuh"

namespace moe_w2 {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Residency table of a step (null table: ids are slots already).
struct SlotMap {
    const int32_t* slot_of;   // [n_route] slot of each routed expert id, < 0 when not resident
    int32_t n_route;
    int32_t* ids_eff;         // [P] slot of each pair, -1 when it is left out (null: not written)
    uint32_t* misses;         // pairs whose expert is not resident (null: not counted)
};

// Bin of a routed id: its slot in [0, E), or E when the pair is left out, with
// `bad` set for an id or slot outside its range and `miss` for a missing expert.
__device__ __forceinline__ int pair_bin(int e, const SlotMap& m, int32_t E, uint32_t& bad, uint32_t& miss)
{
    if (m.slot_of != nullptr) {
        if ((unsigned)e >= (unsigned)m.n_route) {
            bad = 1;
            return E;
        }
        e = __ldg(m.slot_of + e);
        if (e < 0) {
            miss += 1;
            return E;
        }
    }
    if ((unsigned)e >= (unsigned)E) {
        bad = 1;
        return E;
    }
    return e;
}

// Adds the warp's missing pairs to the counter (one atomic per warp).
__device__ __forceinline__ void count_misses(uint32_t miss, const SlotMap& m)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) miss += __shfl_xor_sync(0xffffffffu, miss, o);
    if (m.misses != nullptr && miss != 0 && (threadIdx.x & 31) == 0) atomicAdd(m.misses, miss);
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t r;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(r));
    return r;
}

// The whole permutation of a step of at most 32 pairs by one warp (lane p holds
// pair p): the same outputs as the CTA path below, without its barriers.  Bins:
// expert id, E for out-of-range ids, E + 1 for lanes past P (never stored).
// Returns the number of valid pairs (to every lane).
__device__ int warp_permute(const int32_t* __restrict__ ids, const SlotMap& map, int32_t P, int32_t E,
                            int32_t* __restrict__ sorted, int32_t* __restrict__ inv, int32_t* __restrict__ offsets,
                            int32_t* __restrict__ active, int32_t* __restrict__ active_count,
                            int4* __restrict__ tiles, int32_t* __restrict__ tile_count, int32_t tile_rows,
                            int* s_bin, uint32_t* status)
{
    const int lane = threadIdx.x & 31;
    int b = E + 1;
    uint32_t bad = 0, miss = 0;
    if (lane < P) {
        b = pair_bin(__ldg(ids + lane), map, E, bad, miss);
        if (map.ids_eff != nullptr) map.ids_eff[lane] = b < E ? b : -1;
    }
    if (__any_sync(0xffffffffu, bad != 0) && lane == 0) flag_status(status, MOE_W2_DEV_BAD_EXPERT_ID);
    count_misses(miss, map);
    // stable rank inside the bin, and the pairs of lower bins
    const uint32_t same = __match_any_sync(0xffffffffu, b);
    const int rank = __popc(same & lanemask_lt());
    const bool lead = rank == 0 && b < E;   // first pair of an active expert
    const int cnt = __popc(same);
    const int ntl = lead && tiles != nullptr ? (cnt + tile_rows - 1) / tile_rows : 0;
    int less = 0, act_before = 0, tiles_before = 0;
    for (int i = 0; i < 32; ++i) {
        const int bi = __shfl_sync(0xffffffffu, b, i);
        const int li = __shfl_sync(0xffffffffu, (int)lead, i);
        const int ti = __shfl_sync(0xffffffffu, ntl, i);
        less += bi < b;
        act_before += (li && bi < b);
        tiles_before += (li && bi < b) ? ti : 0;
    }
    const int pos = less + rank;
    if (lane < P) {
        sorted[pos] = lane;
        inv[lane] = pos;
        s_bin[pos] = b;
    }
    __syncwarp();
    const int sb = lane < P ? s_bin[lane] : E + 1;   // bins in sorted order, nondecreasing
    // offsets[bin] = sorted bins below bin (a binary search over the warp's 32)
    const int last = __shfl_sync(0xffffffffu, sb, 31);
    for (int base = 0; base <= E; base += 32) {
        const int bin = base + lane;
        int lo = 0;
#pragma unroll
        for (int st = 16; st >= 1; st >>= 1)
            if (__shfl_sync(0xffffffffu, sb, lo + st - 1) < bin) lo += st;
        if (last < bin) lo = 32;
        if (bin <= E) offsets[bin] = lo;
    }
    const int n_valid = __popc(__ballot_sync(0xffffffffu, lane < P && b < E));
    if (active != nullptr) {
        if (lead) active[act_before] = b;
        const int n_act = __popc(__ballot_sync(0xffffffffu, lead));
        if (lane == 0) *active_count = n_act;
    }
    if (tiles != nullptr) {
        for (int i = 0; i < ntl; ++i) {
            const int r0 = (int)(((int64_t)i * cnt) / ntl), r1 = (int)(((int64_t)(i + 1) * cnt) / ntl);
            tiles[tiles_before + i] = make_int4(b, less + r0, r1 - r0, 0);
        }
        int tot = ntl;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) *tile_count = tot;
    }
    return n_valid;
}

// Exclusive scan over the CTA of three ints per thread at once (one pass of
// shuffles and two barriers for all three); tot[] receives the three totals.
__device__ int3 cta_exclusive_scan3(int3 v, int3* warp_tmp, int3* tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int3 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yx = __shfl_up_sync(0xffffffffu, x.x, o);
        const int yy = __shfl_up_sync(0xffffffffu, x.y, o);
        const int yz = __shfl_up_sync(0xffffffffu, x.z, o);
        if (lane >= o) {
            x.x += yx;
            x.y += yy;
            x.z += yz;
        }
    }
    if (lane == 31) warp_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int3 w = warp_tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(0xffffffffu, w.x, o);
            const int yy = __shfl_up_sync(0xffffffffu, w.y, o);
            const int yz = __shfl_up_sync(0xffffffffu, w.z, o);
            if (lane >= o) {
                w.x += yx;
                w.y += yy;
                w.z += yz;
            }
        }
        warp_tmp[lane] = w;
    }
    __syncthreads();
    const int3 base = warp ? warp_tmp[warp - 1] : make_int3(0, 0, 0);
    *tot = warp_tmp[kWarps - 1];
    return make_int3(base.x + x.x - v.x, base.y + x.y - v.y, base.z + x.z - v.z);
}

// x [rows][H] -> x_t16 [rows][H]: 4x4 transpose inside each group of 16 (the
// mma.sync decode kernel reads activation rows in this order).
__device__ __forceinline__ void t16_group(const uint16_t* src, uint16_t* dst)
{
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(src + 8));
    // natural words: a.x=(x0,x1) a.y=(x2,x3) a.z=(x4,x5) a.w=(x6,x7) b.x=(x8,x9) ...
    uint4 o, p;
    o.x = __byte_perm(a.x, a.z, 0x5410);  // (x0, x4)
    o.y = __byte_perm(b.x, b.z, 0x5410);  // (x8, x12)
    o.z = __byte_perm(a.x, a.z, 0x7632);  // (x1, x5)
    o.w = __byte_perm(b.x, b.z, 0x7632);  // (x9, x13)
    p.x = __byte_perm(a.y, a.w, 0x5410);  // (x2, x6)
    p.y = __byte_perm(b.y, b.w, 0x5410);  // (x10, x14)
    p.z = __byte_perm(a.y, a.w, 0x7632);  // (x3, x7)
    p.w = __byte_perm(b.y, b.w, 0x7632);  // (x11, x15)
    *reinterpret_cast<uint4*>(dst) = o;
    *reinterpret_cast<uint4*>(dst + 8) = p;
}

// Two elements of a 32-element block of token t, one of 16 threads of the block
// (lanes 16c..16c+15 of a warp hold block c of the warp): byte r of the block in
// each of the token's kActDigits digit rows of xd (packed positions 2r and 2r+1,
// in the fp4_elem order), and from thread 0 the rows' UE8M0 bytes in sxd.
__device__ __forceinline__ void x_digits(const uint16_t* __restrict__ x, int64_t blk, int r, bool live, int32_t H,
                                         uint8_t* __restrict__ xd, uint8_t* __restrict__ sxd)
{
    const int bpr = H / 32;
    const int64_t t = blk / bpr;
    const int c = (int)(blk % bpr);
    float v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int pos = 2 * r + h;
        const int e = (pos & 16) | fp4_elem(pos & 15);
        v[h] = live ? __uint_as_float((uint32_t)__ldg(x + t * H + c * 32 + e) << 16) : 0.f;
    }
#pragma unroll
    for (int d = 0; d < kActDigits; ++d) {
        // the block's largest leftover over the 16 threads of the block
        float amax = fmaxf(fabsf(v[0]), fabsf(v[1]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const uint32_t s = digit_scale_byte(amax);
        const float inv = digit_inv_scale(s), sc = digit_scale(s);
        float q0, q1;
        const uint32_t nn = e2m1x2_digits_hw(v[0] * inv, v[1] * inv, q0, q1);
        v[0] -= q0 * sc;
        v[1] -= q1 * sc;
        if (live) {
            xd[(kActDigits * t + d) * (H / 2) + c * 16 + r] = (uint8_t)nn;
            if (r == 0) sxd[(kActDigits * t + d) * bpr + c] = (uint8_t)s;
        }
    }
}

__global__ void __launch_bounds__(kThreads) permute_kernel(
    const int32_t* __restrict__ ids, const SlotMap map, int32_t P, int32_t E, int32_t* __restrict__ sorted,
    int32_t* __restrict__ inv, int32_t* __restrict__ offsets, int32_t* __restrict__ active,
    int32_t* __restrict__ active_count, int4* __restrict__ tiles, int32_t* __restrict__ tile_count,
    int32_t tile_rows, const uint16_t* __restrict__ x, uint16_t* __restrict__ x_t16, uint8_t* __restrict__ xd,
    uint8_t* __restrict__ sxd, int32_t H, int64_t n_blocks, int32_t* __restrict__ counters, int32_t n_counters,
    uint16_t* __restrict__ y, int64_t y_elems, uint32_t* status)
{
    // the decode layer kernel may launch now; it waits for this grid to finish
    // before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;");
    if (blockIdx.x > 0 && x_t16 != nullptr) {
        // extra CTAs: x in T16 order for the mma.sync decode kernel
        const int64_t n_groups = n_blocks * 2;
        const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
        for (int64_t g = (int64_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x; g < n_groups; g += stride)
            t16_group(x + g * 16, x_t16 + g * 16);
        return;
    }
    if (blockIdx.x > 0) {
        // extra CTAs: the block-scaled decode kernel's digit rows of every
        // token, 16 threads per 32-element block (warp-uniform trip count)
        const int64_t stride = (int64_t)(gridDim.x - 1) * (blockDim.x / 16);
        const int64_t nb_pad = (n_blocks + 1) & ~(int64_t)1;
        for (int64_t b = (int64_t)(blockIdx.x - 1) * (blockDim.x / 16) + (threadIdx.x >> 4); b < nb_pad; b += stride)
            x_digits(x, b < n_blocks ? b : 0, threadIdx.x & 15, b < n_blocks, H, xd, sxd);
        return;
    }
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
    if (P <= 32) {
        // a small step: one warp permutes; the CTA zeroes y if no pair is valid
        __shared__ int s_bin[32];
        __shared__ int s_valid;
        if (threadIdx.x < 32) {
            const int n_valid = warp_permute(ids, map, P, E, sorted, inv, offsets, active, active_count, tiles,
                                             tile_count, tile_rows, s_bin, status);
            if (threadIdx.x == 0) s_valid = n_valid;
        }
        __syncthreads();
        if (y != nullptr && s_valid == 0)
            for (int64_t i = threadIdx.x; i < y_elems; i += kThreads) y[i] = 0;
        return;
    }
    extern __shared__ int32_t smem[];
    __shared__ int3 warp_tmp[kWarps];
    int3 sh_tot;   // totals of the fused scan (same value in every thread)
    const int nb = E + 1;                 // bin E collects the pairs left out
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // slices of 32-pair multiples, one per warp; only as many as P needs
    const int chunk = (((P + kWarps - 1) / kWarps) + 31) & ~31;
    const int n_slices = chunk ? (P + chunk - 1) / chunk : 0;
    int32_t* cnt = smem;                    // [n_slices][nb] counts, then write cursors
    int32_t* soff = smem + kWarps * nb;     // [nb] per-expert totals, then exclusive offsets

    for (int i = tid; i < n_slices * nb; i += kThreads) cnt[i] = 0;
    __syncthreads();

    const int p0 = warp * chunk;
    const int p1 = min(P, p0 + chunk);
    uint32_t bad = 0, miss = 0;

    // pass 1: counts per (slice, expert)
    for (int pb = p0; pb < p1; pb += 32 * 8) {
        int e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int p = pb + u * 32 + lane;
            e[u] = (p < p1) ? __ldg(ids + p) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int p = pb + u * 32 + lane;
            if (p >= p1) continue;
            const int b = pair_bin(e[u], map, E, bad, miss);
            if (map.ids_eff != nullptr) map.ids_eff[p] = b < E ? b : -1;
            atomicAdd(&cnt[warp * nb + b], 1);
        }
    }
    count_misses(miss, map);
    __syncthreads();

    // per-expert totals; cnt becomes the exclusive prefix over slices
    for (int b = tid; b < nb; b += kThreads) {
        int run = 0;
        for (int w = 0; w < n_slices; ++w) {
            int c = cnt[w * nb + b];
            cnt[w * nb + b] = run;
            run += c;
        }
        soff[b] = run;
    }
    __syncthreads();

    // one fused scan over bins (two bins per thread covers nb <= 2048) of
    // (pairs, active flags, tiles)
    const int b0 = 2 * tid, b1 = 2 * tid + 1;
    const int t0 = (b0 < nb) ? soff[b0] : 0, t1 = (b1 < nb) ? soff[b1] : 0;
    const int f0 = (b0 < E && t0 > 0), f1 = (b1 < E && t1 > 0);
    const int n0 = (tiles != nullptr && b0 < E) ? (t0 + tile_rows - 1) / tile_rows : 0;
    const int n1 = (tiles != nullptr && b1 < E) ? (t1 + tile_rows - 1) / tile_rows : 0;
    const int3 ex = cta_exclusive_scan3(make_int3(t0 + t1, f0 + f1, n0 + n1), warp_tmp, &sh_tot);
    if (b0 < nb) { soff[b0] = ex.x; offsets[b0] = ex.x; }
    if (b1 < nb) { soff[b1] = ex.x + t0; offsets[b1] = ex.x + t0; }
    if (active != nullptr) {
        if (f0) active[ex.y] = b0;
        if (f1) active[ex.y + f0] = b1;
        if (tid == 0) *active_count = sh_tot.y;
    }
    if (tiles != nullptr) {
        for (int i = 0; i < n0; ++i) {
            int r0 = (int)(((int64_t)i * t0) / n0), r1 = (int)(((int64_t)(i + 1) * t0) / n0);
            tiles[ex.z + i] = make_int4(b0, ex.x + r0, r1 - r0, 0);
        }
        for (int i = 0; i < n1; ++i) {
            int r0 = (int)(((int64_t)i * t1) / n1), r1 = (int)(((int64_t)(i + 1) * t1) / n1);
            tiles[ex.z + n0 + i] = make_int4(b1, ex.x + t0 + r0, r1 - r0, 0);
        }
        if (tid == 0) *tile_count = sh_tot.z;
    }
    __syncthreads();
    // no valid pair at all (offset of the invalid-id bin is 0): nothing will
    // write y, so it is zeroed here
    if (y != nullptr && soff[E] == 0)
        for (int64_t i = tid; i < y_elems; i += kThreads) y[i] = 0;

    // write cursors = expert offset + prefix over earlier slices
    for (int w = 0; w < n_slices; ++w)
        for (int b = tid; b < nb; b += kThreads) cnt[w * nb + b] += soff[b];
    __syncthreads();

    // pass 2: stable scatter
    const uint32_t lt = lanemask_lt();
    for (int pb = p0; pb < p1; pb += 32 * 8) {
        int e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            int p = pb + u * 32 + lane;
            e[u] = (p < p1) ? __ldg(ids + p) : 0;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (pb + u * 32 >= p1) break;   // warp-uniform
            const int p = pb + u * 32 + lane;
            const bool valid = p < p1;
            uint32_t bad2 = 0, miss2 = 0;   // counted in pass 1
            const int b = valid ? pair_bin(e[u], map, E, bad2, miss2) : E;
            const int key = valid ? b : (nb + lane);
            const uint32_t mask = __match_any_sync(0xffffffffu, key);
            const int rank = __popc(mask & lt);
            int pos = 0;
            if (valid) pos = cnt[warp * nb + b] + rank;
            __syncwarp();
            if (valid) {
                sorted[pos] = p;
                inv[p] = pos;
                if (rank == 0) cnt[warp * nb + b] += __popc(mask);
            }
            __syncwarp();
        }
    }
    if (bad) flag_status(status, MOE_W2_DEV_BAD_EXPERT_ID);
}

}  // namespace

cudaError_t launch_permute(const int32_t* ids, const PermuteSlots& slots, int32_t T, int32_t k, int32_t E,
                           int32_t* sorted, int32_t* inv, int32_t* offsets, int32_t* active, int32_t* active_count,
                           int4* tiles, int32_t* tile_count, int32_t tile_rows, const uint16_t* x, uint16_t* x_t16,
                           uint8_t* xd, uint8_t* sxd, int32_t H, int32_t* counters, int32_t n_counters, uint16_t* y,
                           uint32_t* status, cudaStream_t s)
{
    const int32_t P = T * k;
    const size_t smem = sizeof(int32_t) * (size_t)(kWarps + 1) * (E + 1);
    static bool ready[kMaxDevices];
    int dev = 0;
    cudaError_t e0 = once_per_device(ready, dev, [](int) {
        return cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(sizeof(int32_t) * (kWarps + 1) * (MOE_W2_MAX_EXPERTS + 1)));
    });
    if (e0 != cudaSuccess) return e0;
    int64_t n_blocks = 0;
    int extra = 0;
    if (x != nullptr && x_t16 != nullptr) {
        n_blocks = (int64_t)T * H / 32;
        extra = (int)std::min<int64_t>((n_blocks * 2 + kThreads - 1) / kThreads, 4 * (int64_t)sm_count());
    } else if (x != nullptr && xd != nullptr) {
        n_blocks = (int64_t)T * H / 32;
        extra = (int)std::min<int64_t>((n_blocks * 16 + kThreads - 1) / kThreads, 4 * (int64_t)sm_count());
    }
    const SlotMap map{slots.slot_of, slots.n_route, slots.ids_eff, slots.misses};
    permute_kernel<<<1 + extra, kThreads, smem, s>>>(ids, map, P, E, sorted, inv, offsets, active, active_count, tiles,
                                                     tile_count, tile_rows, x, x_t16, xd, sxd, H, n_blocks,
                                                     counters, n_counters, y, y ? (int64_t)T * H : 0, status);
    return cudaGetLastError();
}

}  // namespace moe_w2
