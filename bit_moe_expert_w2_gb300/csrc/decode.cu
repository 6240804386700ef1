// Decode path (T <= 64): the 2-bit planes of every active expert are streamed
// from HBM once per layer, expanded in registers and fed to tensor-core MMAs.
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": codes expanded in
// registers through a byte-permute lookup table and fed to tensor-core MMAs;
// section "FP4 recovery": decode is HBM-bound, the 2-bit read is the cost.  Page
// "The v0.24.0 port", section "Benchmarks": tokens grouped by expert, so each
// active expert's weights are read once per step however many tokens use it.
// Page "The v0.24.0 port", "Deterministic unpermute" bullet: per-pair results
// are placed in their own slot and summed over top_k in a fixed order.
//
// Why mma.sync here and not tcgen05: with N = a handful of pairs, every
// tcgen05.mma (M=128, K=16) of a CTA costs ~105 cycles whatever N is (measured
// on GB300), which caps a CTA far below HBM rate, while mma.sync m16n8k16 keeps
// the weights in registers and reaches the full tensor rate with enough warps.
// The expansion is integer work split over two pipes: per 16-code word two
// masks and eight byte-permutes on the ALU pipe, and the eight selector words as
// multiply-adds on the FMA pipe (the multipliers are kernel parameters, so they
// stay multiply-adds instead of becoming ALU shifts).  Codes stream through a
// per-warp cp.async ring (3 chunks deep).
//
// Per 256-wide K chunk a row is 64 code bytes; thread c of a quad owns bytes
// [16c, 16c+16), i.e. four 16-code words; MMA (word i, r) takes codes (r, r+4)
// and (r+8, r+12) of word i from every thread of the quad, which is what the
// T16 activation layout stores next to each other (one 64-bit load per B
// fragment).
//
// Work item = (tile of <= 16 pairs of one expert, 32 weight rows).  A warp holds
// two m16 tiles; the four warps of a CTA split K and reduce in shared memory in
// warp order.  gate_up: m-tile t = gate rows n0+8t.. (A rows 0-7) and the
// matching up rows (A rows 8-15), so gate and up of one (row, pair) meet in one
// thread for the SiLU(gate)*up epilogue.  down: 32 consecutive rows of W_down;
// the epilogue multiplies by the router weight and writes the pair's fp32 slot;
// the last CTA to finish a 32-row block of y sums the k slots of every token in
// j order and writes y (counter per row block, reset by the permutation kernel).
#include <algorithm>

#include "tc.cuh"

namespace moe_w2 {

namespace {

#ifndef MOE_W2_DEC_MIN_CTAS
#define MOE_W2_DEC_MIN_CTAS 4        // CTAs per SM the register budget is sized for
#endif
constexpr int kChunk = 256;   // K elements per chunk
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxNT = 2;     // n-tiles of 8 pairs per item (tiles of <= 16 pairs)

struct DecArgs {
    const uint8_t* codes;      // [E][rows_per_expert][K/4]
    const uint8_t* scales;     // [E][rows_per_expert][K/32]
    int32_t K;
    int32_t rows_per_expert;
    int32_t I;
    int32_t H;
    int32_t T;
    int32_t k;
    int32_t E;
    int32_t row_blocks;
    const int4* tiles;
    const int32_t* tile_count;
    const int32_t* sorted;
    const float* weights;
    const int32_t* ids;
    const uint16_t* act;       // B rows: x_t16 per token (gate_up) or h_t16 per pair (down)
    uint16_t* h_t16;           // gate_up output [P][I]
    float* stage;              // down output [P][H]
    int32_t* counters;         // down: per 32-row block of y
    uint16_t* y;
    uint32_t* status;
};

// Coherent 128-bit load (plain ld.global) for data another CTA of the same
// launch wrote: the reader's CTA observed the writer's release with a GPU-scope
// acquire followed by a CTA barrier, so these loads see the data.  The
// non-coherent read-only path (ld.global.nc) is not allowed for it.
__device__ __forceinline__ uint4 ldg_coherent_u4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ld_acquire(const int32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t word_of(const uint4& q, int i)
{
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// Per-thread asynchronous copies global -> shared; the issuing thread's
// wait_group plus a warp barrier orders them before the warp reads them back.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a) : "memory");
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a) : "memory");
    return r;
}
__device__ __forceinline__ uint32_t lds8(uint32_t a)
{
    uint32_t r;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(r) : "r"(a) : "memory");
    return r;
}

// Per-warp ring of kDepth chunks.  Slot layout: codes [row a][lane] 16 bytes
// (lane-major, so a warp's 128-bit reads are conflict-free), then scales
// [row a][g] the chunk's 8 UE8M0 bytes of the quad's row (copied by lane c = 0;
// thread c reads bytes 2c and 2c+1).
constexpr int kDepth = 3;
constexpr uint32_t kRingCodeBytes = 4 * 32 * 16;   // per slot
constexpr uint32_t kRingScaleBytes = 4 * 8 * 8;
constexpr uint32_t kRingSlot = kRingCodeBytes + kRingScaleBytes;
constexpr uint32_t kRingWarp = kDepth * kRingSlot;

template <bool kGateUp, int NT>
__device__ __forceinline__ void run_item(const DecArgs& p, const SelConst& k, uint32_t lut_base,
                                         float (*red)[2][kMaxNT][32][4], uint32_t ring_base, int e, int q0,
                                         int nrows, int rb, uint32_t& lut_and)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int nch = p.K / kChunk;
    const int64_t rowb = p.K / 4, srowb = p.K / 32;

    // the thread's four A rows: m-tile 0 -> (g, g+8), m-tile 1 -> (16+g, 24+g)
    int64_t row[4];
    if (kGateUp) {
        const int64_t base = (int64_t)e * p.rows_per_expert + rb * 16;
        row[0] = base + g;            // gate n0+g
        row[1] = base + p.I + g;      // up   n0+g
        row[2] = base + 8 + g;        // gate n0+8+g
        row[3] = base + p.I + 8 + g;  // up   n0+8+g
    } else {
        const int64_t base = (int64_t)e * p.rows_per_expert + rb * 32;
        row[0] = base + g;
        row[1] = base + 8 + g;
        row[2] = base + 16 + g;
        row[3] = base + 24 + g;
    }
    // global sources of this warp's first chunk; each later chunk is kWarps chunks on
    const uint8_t* cp[4];
    const uint8_t* sp[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        cp[a] = p.codes + row[a] * rowb + warp * 64 + c * 16;
        sp[a] = p.scales + row[a] * srowb + warp * 8;
    }
    // B rows: pair j = 8*nt + g of the tile.  Columns past the tile's pairs read
    // pair 0's row (always valid); their results are never stored.
    const uint16_t* brow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int j = nt * 8 + g < nrows ? nt * 8 + g : 0;
        const int64_t br = kGateUp ? (int64_t)(__ldg(p.sorted + q0 + j) / p.k) : (int64_t)(q0 + j);
        brow[nt] = p.act + br * p.K + warp * kChunk + c * 64;
    }

    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;

    // ring of this warp's chunks ch = warp + kWarps * idx
    const uint32_t ring = ring_base + (uint32_t)warp * kRingWarp;
    const int my_chunks = nch > warp ? (nch - warp + kWarps - 1) / kWarps : 0;
    uint32_t wr_slot = ring;
    int issued = 0;
    auto issue = [&]() {
        if (issued < my_chunks) {
            const int64_t off = (int64_t)issued * (kWarps * 64);
#pragma unroll
            for (int a = 0; a < 4; ++a) cp_async16(wr_slot + (uint32_t)(a * 32 + lane) * 16, cp[a] + off);
            if (c == 0) {
#pragma unroll
                for (int a = 0; a < 4; ++a)
                    cp_async8(wr_slot + kRingCodeBytes + (uint32_t)(a * 8 + g) * 8, sp[a] + (int64_t)issued * (kWarps * 8));
            }
        }
        cp_async_commit();
        ++issued;
        wr_slot = wr_slot + kRingSlot == ring + kRingWarp ? ring : wr_slot + kRingSlot;
    };
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d) issue();
    uint32_t rd_slot = ring;
    for (int idx = 0; idx < my_chunks; ++idx) {
        issue();
        cp_async_wait<kDepth - 1>();
        __syncwarp();
        uint4 q[4];
        uint2 L[4][2];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            q[a] = lds128(rd_slot + (uint32_t)(a * 32 + lane) * 16);
            const uint32_t sa = rd_slot + kRingCodeBytes + (uint32_t)(a * 8 + g) * 8 + 2 * c;
            L[a][0] = lds64(lut_base + lds8(sa) * 8u);
            L[a][1] = lds64(lut_base + lds8(sa + 1) * 8u);
            lut_and &= L[a][0].x & L[a][1].x;
        }
        const uint16_t* bsrc[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) bsrc[nt] = brow[nt] + (int64_t)idx * (kWarps * kChunk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 B0[NT], B1[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kGateUp) {   // x in T16 order, written by an earlier launch
                    B0[nt] = ldg_u4(bsrc[nt] + i * 16);
                    B1[nt] = ldg_u4(bsrc[nt] + i * 16 + 8);
                } else {         // h, written by the gate_up items of this launch
                    B0[nt] = ldg_coherent_u4(bsrc[nt] + i * 16);
                    B1[nt] = ldg_coherent_u4(bsrc[nt] + i * 16 + 8);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const Masks ma = word_masks(word_of(q[2 * mt], i), k), mb = word_masks(word_of(q[2 * mt + 1], i), k);
                const uint2 la = L[2 * mt][i >> 1], lb = L[2 * mt + 1][i >> 1];
                uint32_t alo[4], ahi[4], blo[4], bhi[4];
                selectors(ma, k, alo, ahi);
                selectors(mb, k, blo, bhi);
                uint32_t afrag[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    afrag[r][0] = prmt(la.x, la.y, alo[r]);
                    afrag[r][1] = prmt(lb.x, lb.y, blo[r]);
                    afrag[r][2] = prmt(la.x, la.y, ahi[r]);
                    afrag[r][3] = prmt(lb.x, lb.y, bhi[r]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint4& Bv = (r < 2) ? B0[nt] : B1[nt];
                        mma_bf16_16816(acc[mt][nt], afrag[r], (r & 1) ? Bv.z : Bv.x, (r & 1) ? Bv.w : Bv.y);
                    }
            }
        }
        __syncwarp();
        rd_slot = rd_slot + kRingSlot == ring + kRingWarp ? ring : rd_slot + kRingSlot;
    }
    cp_async_wait<0>();

    // split-K reduction in warp order
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int v = 0; v < 4; ++v) red[warp][mt][nt][lane][v] = acc[mt][nt][v];
    __syncthreads();
    // warp w finalises m-tile (w & 1), n-tile (w >> 1)
    const int mt = warp & 1;
    for (int nt = warp >> 1; nt < NT; nt += 2) {
        float v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[w][mt][nt][lane][q];
            v[q] = s;
        }
        if (kGateUp) {
            const int pos = t16_pos(rb * 16 + mt * 8 + g);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = nt * 8 + 2 * c + h;
                if (j < nrows) {
                    __nv_bfloat16 hb = __float2bfloat16_rn(silu_f(v[h]) * v[2 + h]);
                    p.h_t16[(int64_t)(q0 + j) * p.I + pos] = *reinterpret_cast<uint16_t*>(&hb);
                }
            }
        } else {
            const int m = rb * 32 + mt * 16 + g;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = nt * 8 + 2 * c + h;
                if (j < nrows) {
                    const int pr = __ldg(p.sorted + q0 + j);
                    const float wt = __ldg(p.weights + pr);
                    p.stage[(int64_t)pr * p.H + m] = wt * v[h];
                    p.stage[(int64_t)pr * p.H + m + 8] = wt * v[2 + h];
                }
            }
        }
    }
    __syncthreads();
}

// One persistent, co-resident grid runs the whole decode layer.  Items come
// from one queue: indices [0, n_gu) are gate_up items (tile, 16 gate + 16 up
// rows), [n_gu, n_gu + n_dn) down items (tile, 32 rows of y).  CTA c starts with
// item c and then takes the next free index from a global counter (taken one
// item ahead, so the atomic's latency hides behind the current item); a CTA
// that runs out of gate_up work moves straight on to down work.  A down item of
// tile t needs h of every row of t, so it waits until the tile's gate_up counter
// reaches the number of gate_up row blocks.  Every gate_up index is handed out
// before any down index and all CTAs are resident at once (cooperative launch),
// so the waits always end; each is still bounded and gives up with the
// pipeline-timeout status bit.  Which CTA runs an item never changes its result.
__global__ void __launch_bounds__(kThreads, MOE_W2_DEC_MIN_CTAS)
decode_layer_kernel(DecArgs gu, DecArgs dn, int32_t* __restrict__ gu_done, int32_t* __restrict__ queue)
{
    __shared__ uint2 lut[256];
    __shared__ float red[kWarps][2][kMaxNT][32][4];
    __shared__ int last_flag;
    __shared__ int abort_flag;
    __shared__ int next_item;
    extern __shared__ __align__(16) uint8_t ring_smem[];   // kWarps * kRingWarp bytes
    const uint32_t ring_base = (uint32_t)__cvta_generic_to_shared(ring_smem);
    const uint32_t lut_base = (uint32_t)__cvta_generic_to_shared(lut);
    for (int s = threadIdx.x; s < 256; s += kThreads) {
        ScaleLut l = make_lut((uint32_t)s);
        lut[s] = make_uint2(l.lut, l.lo);
    }
    if (threadIdx.x == 0) abort_flag = 0;
    const SelConst k = sel_const_regs();
    __syncthreads();

    const int n_tiles = *gu.tile_count;
    const int n_gu = n_tiles * gu.row_blocks;
    const int n_all = n_gu + n_tiles * dn.row_blocks;
    // AND of every lut word used: a valid scale's lut word has bit 31 set, an
    // invalid one is 0, so the AND is 0 exactly when a bad scale byte was read.
    uint32_t lut_and = 0xFFFFFFFFu;

    int it = blockIdx.x;
    while (it < n_all) {
        // the item after this one (read after the barriers of this item)
        if (threadIdx.x == 0) next_item = (int)gridDim.x + atomicAdd(queue, 1);
        if (it < n_gu) {
            // gate_up: h = SiLU(gate) * up
            const int ti = it / gu.row_blocks;
            const int4 tile = gu.tiles[ti];
            const int rb = it % gu.row_blocks;
            if (tile.z <= 8) run_item<true, 1>(gu, k, lut_base, red, ring_base, tile.x, tile.y, tile.z, rb, lut_and);
            else run_item<true, 2>(gu, k, lut_base, red, ring_base, tile.x, tile.y, tile.z, rb, lut_and);
            // run_item ends with a CTA barrier after its h stores
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(gu_done + ti, 1);
            }
        } else {
            // down (+ combine): stage slot = w * (W_down h)
            const int id = it - n_gu;
            const int ti = id / dn.row_blocks;
            const int4 tile = dn.tiles[ti];
            const int rb = id % dn.row_blocks;
            if (threadIdx.x == 0 && (int)ld_acquire(gu_done + ti) < gu.row_blocks) {
                const long long t0 = clock64();
                while ((int)ld_acquire(gu_done + ti) < gu.row_blocks) {
                    if (clock64() - t0 > kWaitLimitCycles) {
                        abort_flag = 1;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            __syncthreads();
            if (abort_flag) {
                if (threadIdx.x == 0) flag_status(dn.status, kDevPipelineTimeout);
                break;
            }
            if (tile.z <= 8) run_item<false, 1>(dn, k, lut_base, red, ring_base, tile.x, tile.y, tile.z, rb, lut_and);
            else run_item<false, 2>(dn, k, lut_base, red, ring_base, tile.x, tile.y, tile.z, rb, lut_and);
            // The last of the n_tiles items that wrote rows [32 rb, 32 rb + 32) of
            // the pair slots sums them into y (fixed j order per token).
            __threadfence();
            if (threadIdx.x == 0) last_flag = (atomicAdd(dn.counters + rb, 1) == n_tiles - 1);
            __syncthreads();
            if (last_flag) {
                __threadfence();
                for (int i = threadIdx.x; i < dn.T * 32; i += kThreads) {
                    const int t = i >> 5, m = rb * 32 + (i & 31);
                    float s = 0.f;
                    for (int j = 0; j < dn.k; ++j) {
                        const int ej = __ldg(dn.ids + t * dn.k + j);
                        if ((unsigned)ej < (unsigned)dn.E) s += __ldcg(dn.stage + (int64_t)(t * dn.k + j) * dn.H + m);
                    }
                    __nv_bfloat16 yb = __float2bfloat16_rn(s);
                    dn.y[(int64_t)t * dn.H + m] = *reinterpret_cast<uint16_t*>(&yb);
                }
                if (threadIdx.x == 0) dn.counters[rb] = 0;
            }
            __syncthreads();
        }
        it = next_item;
        __syncthreads();   // everyone has read next_item before thread 0 overwrites it
    }
    if (lut_and == 0) flag_status(gu.status, MOE_W2_DEV_BAD_SCALE);
}

}  // namespace

cudaError_t launch_decode(const uint16_t* x, const int32_t* ids, const float* weights, const moe_w2_planes& w,
                          int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                          const PhaseEvents& ev)
{
    (void)x;
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    constexpr int kDyn = kWarps * kRingWarp;
    static int occ = 0;
    if (occ == 0) {
        cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_layer_kernel, kThreads, kDyn);
        if (e != cudaSuccess) return e;
        occ = std::max(occ, 1);
    }
    const int64_t tiles = max_tiles(P, E, true);

    DecArgs gp{};
    gp.codes = w.w13_codes;
    gp.scales = w.w13_scales;
    gp.K = H;
    gp.rows_per_expert = 2 * I;
    gp.I = I;
    gp.H = H;
    gp.T = T;
    gp.k = k;
    gp.E = E;
    gp.row_blocks = I / 16;
    gp.tiles = ws.tiles;
    gp.tile_count = ws.tile_count;
    gp.sorted = ws.sorted;
    gp.weights = weights;
    gp.ids = ids;
    gp.act = ws.xa;
    gp.h_t16 = ws.h;
    gp.stage = ws.stage;
    gp.counters = ws.counters;
    gp.y = y;
    gp.status = status;

    DecArgs dp = gp;
    dp.codes = w.w2_codes;
    dp.scales = w.w2_scales;
    dp.K = I;
    dp.rows_per_expert = H;
    dp.row_blocks = H / 32;
    dp.act = ws.h;
    int32_t* gu_done = ws.counters + H / 32;   // [tiles], zeroed by the permutation kernel
    int32_t* queue = gu_done + tiles;          // item queue, zeroed by the permutation kernel

    // every CTA resident at once: at most occupancy x SMs, and no more than the
    // larger phase has items
    const int64_t grid = std::min<int64_t>((int64_t)sm_count() * occ,
                                           tiles * std::max<int64_t>(gp.row_blocks, dp.row_blocks));
    cudaError_t e = ev.record(1, s);
    if (e != cudaSuccess) return e;
    if ((e = ev.record(2, s)) != cudaSuccess) return e;   // one kernel: phases 1 and 2 coincide
    void* args[] = {&gp, &dp, &gu_done, &queue};
    e = cudaLaunchCooperativeKernel((const void*)decode_layer_kernel, dim3((unsigned)grid), dim3(kThreads), args,
                                    (size_t)kDyn, s);
    return e;
}

}  // namespace moe_w2
