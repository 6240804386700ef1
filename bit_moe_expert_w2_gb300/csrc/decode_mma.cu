// Decode path for the smallest steps (few pairs, see decode_use_mma): the 2-bit
// planes of every active expert are streamed from HBM once per layer, expanded
// to bf16 in registers and fed to mma.sync tensor-core MMAs.
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
// The expansion is integer work on the ALU pipe (two masks, five shifts and
// eight byte-permutes per 16 codes) plus two multiply-adds on the FMA pipe.
//
// One kernel runs the whole layer (gate_up, then down with the combine).  Work
// item = (tile of <= 16 pairs of one expert, 32 weight rows).  Each CTA has four
// consumer warps that split K of an item (256-element chunks, round robin) and
// reduce in shared memory in warp order, and one producer warp that runs ahead
// through the CTA's items: it takes items from a global queue, publishes each
// item's tile through a small shared-memory ring, and streams every chunk's code
// bytes (TMA: 32 rows x 64 bytes) and scale bytes (one 8-byte cp.async per row)
// into a ring of chunk slots.  Consumers only wait on a slot's barrier, read it
// from shared memory and release it, so the loads of the next item overlap the
// end of the current one.
//
// Per 256-wide K chunk a row is 64 code bytes; thread c of a quad owns bytes
// [16c, 16c+16), i.e. four 16-code words; MMA (word i, r) takes codes (r, r+4)
// and (r+8, r+12) of word i from every thread of the quad, which is what the
// T16 activation layout stores next to each other (one 64-bit load per B
// fragment).  gate_up: m-tile t = gate rows n0+8t.. (A rows 0-7) and the
// matching up rows (A rows 8-15), so gate and up of one (row, pair) meet in one
// thread for the SiLU(gate)*up epilogue.  down: 32 consecutive rows of W_down;
// the epilogue multiplies by the router weight and writes the pair's fp32 slot;
// the last CTA to finish a 32-row block of y sums the k slots of every token in
// j order and writes y (counter per row block, reset by the permutation kernel).
//
// The FP4 layer (page "vLLM-Moet wiki", "The kernels" and "FP4 recovery":
// moe_w4_mm, the same forward over the NVFP4 experts at twice the plane bytes)
// is the same kernel with kW4: a chunk row is 128 bytes of e2m1 nibbles and 16
// e4m3 scale bytes (one per 16 elements); thread c of a quad owns the row's
// elements 64c .. 64c+63 as before, and each 16-element block (two words)
// becomes the same bf16 pairs (r, r+4), (r+8, r+12) through fp4_word_bf16 with
// the block's scale folded into the table; scale_2 multiplies the fp32 results
// in the epilogues.
#include <algorithm>
#include <type_traits>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kMinCtasPerSm = 4;     // CTAs per SM the register budget is sized for
constexpr int kChunk = 256;          // K elements per chunk
constexpr int kWarps = 4;            // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;   // + the producer warp
constexpr int kMaxNT = 2;            // n-tiles of 8 pairs per item (tiles of <= 16 pairs)
// Chunk slots: 2-bit planes (kW4 false) or NVFP4 experts (true); both rings
// take the same 36 KB of shared memory.
template <bool kW4> struct Fmt {
    static constexpr int kSlots = kW4 ? 8 : 16;                         // chunk slots
    static constexpr uint32_t kRowBytes = kW4 ? 128 : 64;               // code bytes of a row per chunk
    static constexpr uint32_t kRowScaleBytes = kW4 ? 16 : 8;            // scale bytes of a row per chunk
    static constexpr uint32_t kSlotCodeBytes = 32 * kRowBytes;          // 32 rows
    static constexpr uint32_t kSlotBytes = kSlotCodeBytes + 32 * kRowScaleBytes;   // a multiple of 128
    static constexpr uint32_t kRingBytes = kSlots * kSlotBytes;
    using Lut = std::conditional_t<kW4, uint4, uint2>;
};
constexpr int kInfo = 16;            // published items in flight
constexpr uint32_t kConsumerBarrier = 1;       // named barrier id of the consumer warps

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
    DepWait dep;               // down items' wait for their tile's h: target bias and limit
    const float* scale_2;      // FP4 layer: per-tensor scale_2 of expert e at e * s2_stride (+1: up)
    int32_t s2_stride;
};

template <bool kW4>
struct SharedState {
    uint64_t full[Fmt<kW4>::kSlots];   // producer -> consumers: slot filled (expect_tx arrival + 32 cp.async arrivals)
    uint64_t empty[Fmt<kW4>::kSlots];  // consumer warp -> producer: slot read
    uint64_t info_full[kInfo];  // producer -> consumers: item published
    uint64_t info_empty[kInfo]; // consumer warps -> producer: item finished
    int4 info[kInfo];           // (item index, or -1 at the end; expert; first slot; pairs)
    typename Fmt<kW4>::Lut lut[256];   // per scale byte: ScaleLut words, or the NVFP4 product table
    float red[kWarps][2][kMaxNT][32][4];
    int4 cur_info;              // the item the consumer warps work on
    int last_flag;
    int stop;
    int abort_flag;
};

__device__ __forceinline__ uint32_t ld_acquire(const int32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(kConsumerBarrier), "n"(kWarps * 32) : "memory");
}
__device__ __forceinline__ uint32_t word_of(const uint4& q, int i)
{
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// One item on the consumer warps: K chunks ch = warp, warp + 4, ... from ring
// slots (qbase + ch) % kSlots, then the split-K reduction and the epilogue.
template <bool kGateUp, int NT, bool kW4>
__device__ __forceinline__ void run_item(const DecArgs& p, const SelConst& k, SharedState<kW4>& sh,
                                         const uint8_t* ring, uint32_t qbase, int q0, int nrows, int rb, int expert,
                                         uint32_t& lut_and)
{
    using F = Fmt<kW4>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int nch = p.K / kChunk;
    // slot rows of the thread's four A rows: m-tile 0 -> (g, g+8), m-tile 1 -> (16+g, 24+g);
    // gate_up slot rows 0-15 are gate rows n0.., 16-31 the matching up rows
    int srow[4];
    if (kGateUp) {
        srow[0] = g;
        srow[1] = 16 + g;
        srow[2] = 8 + g;
        srow[3] = 24 + g;
    } else {
        srow[0] = g;
        srow[1] = 8 + g;
        srow[2] = 16 + g;
        srow[3] = 24 + g;
    }
    // B rows: pair j = 8*nt + g of the tile.  Columns past the tile's pairs read
    // pair 0's row (always valid); their results are never stored.
    const uint16_t* brow[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int j = nt * 8 + g < nrows ? nt * 8 + g : 0;
        const int64_t br = kGateUp ? (int64_t)(__ldg(p.sorted + q0 + j) / p.k) : (int64_t)(q0 + j);
        brow[nt] = p.act + br * p.K + c * 64;
    }

    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;

    volatile int* abort = &sh.abort_flag;
    for (int ch = warp; ch < nch; ch += kWarps) {
        const uint32_t q = qbase + (uint32_t)ch;
        const uint32_t slot = q % F::kSlots;
        if (!mbar_wait(smem_u32(&sh.full[slot]), (q / F::kSlots) & 1u, abort)) break;
        // plain (compiler-schedulable) shared loads: the wait above is a compiler barrier
        const uint8_t* sp = ring + slot * F::kSlotBytes;
        if constexpr (kW4) {
            // the row's 32 bytes of this thread (elements 64c..64c+63: four blocks of
            // 16, two words each) and the four blocks' e4m3 bytes
            uint4 qa[4][2];
            uint32_t sw[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                qa[a][0] = *reinterpret_cast<const uint4*>(sp + srow[a] * 128 + c * 32);
                qa[a][1] = *reinterpret_cast<const uint4*>(sp + srow[a] * 128 + c * 32 + 16);
                sw[a] = *reinterpret_cast<const uint32_t*>(sp + F::kSlotCodeBytes + srow[a] * 16 + 4 * c);
                if (e4m3_nan_bytes(sw[a]) != 0u) lut_and = 0u;
            }
            const uint16_t* bsrc[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) bsrc[nt] = brow[nt] + (int64_t)ch * kChunk;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 B0[NT], B1[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (kGateUp) {
                        B0[nt] = __ldg(reinterpret_cast<const uint4*>(bsrc[nt] + i * 16));
                        B1[nt] = __ldg(reinterpret_cast<const uint4*>(bsrc[nt] + i * 16 + 8));
                    } else {
                        B0[nt] = *reinterpret_cast<const uint4*>(bsrc[nt] + i * 16);
                        B1[nt] = *reinterpret_cast<const uint4*>(bsrc[nt] + i * 16 + 8);
                    }
                }
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const uint4& va = qa[2 * mt][i >> 1];
                    const uint4& vb = qa[2 * mt + 1][i >> 1];
                    const uint4 La = sh.lut[(sw[2 * mt] >> (8 * i)) & 0xFFu];
                    const uint4 Lb = sh.lut[(sw[2 * mt + 1] >> (8 * i)) & 0xFFu];
                    // elements 0..7 of the block (word 2 (i % 2)) and 8..15 (the next word)
                    uint32_t a_lo[4], a_hi[4], b_lo[4], b_hi[4];
                    fp4_word_bf16(word_of(va, 2 * (i & 1)), La, a_lo[0], a_lo[1], a_lo[2], a_lo[3]);
                    fp4_word_bf16(word_of(va, 2 * (i & 1) + 1), La, a_hi[0], a_hi[1], a_hi[2], a_hi[3]);
                    fp4_word_bf16(word_of(vb, 2 * (i & 1)), Lb, b_lo[0], b_lo[1], b_lo[2], b_lo[3]);
                    fp4_word_bf16(word_of(vb, 2 * (i & 1) + 1), Lb, b_hi[0], b_hi[1], b_hi[2], b_hi[3]);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const uint32_t afrag[4] = {a_lo[r], b_lo[r], a_hi[r], b_hi[r]};
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint4& Bv = (r < 2) ? B0[nt] : B1[nt];
                            mma_bf16_16816(acc[mt][nt], afrag, (r & 1) ? Bv.z : Bv.x, (r & 1) ? Bv.w : Bv.y);
                        }
                    }
                }
            }
        } else {
        uint4 qw[4];
        uint2 L[4][2];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            qw[a] = *reinterpret_cast<const uint4*>(sp + srow[a] * 64 + c * 16);
            const uint8_t* sb = sp + F::kSlotCodeBytes + srow[a] * 8 + 2 * c;
            L[a][0] = sh.lut[sb[0]];
            L[a][1] = sh.lut[sb[1]];
            lut_and &= L[a][0].x & L[a][1].x;
        }
        const uint16_t* bsrc[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) bsrc[nt] = brow[nt] + (int64_t)ch * kChunk;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 B0[NT], B1[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kGateUp) {   // x in T16 order, written by an earlier launch: read-only path
                    B0[nt] = __ldg(reinterpret_cast<const uint4*>(bsrc[nt] + i * 16));
                    B1[nt] = __ldg(reinterpret_cast<const uint4*>(bsrc[nt] + i * 16 + 8));
                } else {         // h, written by gate_up items of this launch: coherent loads
                    B0[nt] = *reinterpret_cast<const uint4*>(bsrc[nt] + i * 16);
                    B1[nt] = *reinterpret_cast<const uint4*>(bsrc[nt] + i * 16 + 8);
                }
            }
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const Masks ma = word_masks(word_of(qw[2 * mt], i), k), mb = word_masks(word_of(qw[2 * mt + 1], i), k);
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
        }   // 2-bit planes
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
    }

    // split-K reduction in warp order
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int v = 0; v < 4; ++v) sh.red[warp][mt][nt][lane][v] = acc[mt][nt][v];
    consumer_sync();
    // warp w finalises m-tile (w & 1), n-tile (w >> 1)
    const int mt = warp & 1;
    for (int nt = warp >> 1; nt < NT; nt += 2) {
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += sh.red[w][mt][nt][lane][e];
            v[e] = s;
        }
        if (kW4) {
            // the tensors' scale_2: gate rows (accumulator rows g) and up rows (g + 8)
            // of gate_up, or the down rows
            const float s_lo = __ldg(p.scale_2 + (int64_t)expert * p.s2_stride);
            const float s_hi = kGateUp ? __ldg(p.scale_2 + (int64_t)expert * p.s2_stride + 1) : s_lo;
            v[0] *= s_lo;
            v[1] *= s_lo;
            v[2] *= s_hi;
            v[3] *= s_hi;
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
    consumer_sync();
}

// One persistent grid runs the whole decode layer.  Items come from one queue:
// indices [0, n_gu) are gate_up items (tile, 16 gate + 16 up rows), [n_gu, n_all)
// down items (tile, 32 rows of y).  Each CTA's producer warp takes every item,
// the first included, from a global counter, so only CTAs that are running hold
// items.  A down item of tile t needs h of every row of t, so the producer waits
// until the tile's gate_up counter reaches the number of gate_up row blocks
// before it publishes the item; every gate_up index is handed out before any
// down index and is held by a running CTA, so the waits always end (each is
// still bounded and gives up with the pipeline-timeout status bit).  Which CTA
// runs an item never changes its result.
template <bool kW4>
__global__ void __launch_bounds__(kThreads, kMinCtasPerSm)
decode_mma_kernel(const __grid_constant__ CUtensorMap gu_map, const __grid_constant__ CUtensorMap dn_map,
                    DecArgs gu, DecArgs dn, int32_t* __restrict__ gu_done, int32_t* __restrict__ queue)
{
    using F = Fmt<kW4>;
    __shared__ SharedState<kW4> sh;
    extern __shared__ uint8_t dyn_smem[];   // kRingBytes + 128 (aligned below)
    // 128-byte aligned ring; offsetting the shared array itself keeps the
    // pointer in the shared window (plain loads from it compile to shared loads)
    const uint32_t pad = (128u - (smem_u32(dyn_smem) & 127u)) & 127u;
    const uint8_t* ring = dyn_smem + pad;
    const uint32_t ring_addr = smem_u32(dyn_smem) + pad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int s = tid; s < 256; s += kThreads) {
        if constexpr (kW4) {
            sh.lut[s] = make_fp4_lut((uint32_t)s);
        } else {
            ScaleLut l = make_lut((uint32_t)s);
            sh.lut[s] = make_uint2(l.lut, l.lo);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < F::kSlots; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1 + 32);
            mbar_init(smem_u32(&sh.empty[s]), 1);
        }
        for (int s = 0; s < kInfo; ++s) {
            mbar_init(smem_u32(&sh.info_full[s]), 1);
            mbar_init(smem_u32(&sh.info_empty[s]), kWarps);
        }
        sh.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    volatile int* abort = &sh.abort_flag;

    // Launched as a programmatic dependent of the permutation kernel: the setup
    // above overlaps it; everything it writes (tiles, counters, x in T16 order)
    // is read only after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int n_tiles = *gu.tile_count;
    const int n_gu = n_tiles * gu.row_blocks;
    const int n_all = n_gu + n_tiles * dn.row_blocks;

    if (warp == kWarps) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            prefetch_tmap(&gu_map);
            prefetch_tmap(&dn_map);
        }
        uint32_t q = 0;
        int it = 0;
        if (lane == 0) it = atomicAdd(queue, 1);
        it = __shfl_sync(0xffffffffu, it, 0);
        for (int n = 0;; ++n) {
            const uint32_t islot = (uint32_t)n % kInfo;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&sh.info_empty[islot]), ((uint32_t)(n / kInfo) & 1u) ^ 1u, abort);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (it >= n_all) {
                if (lane == 0) {
                    sh.info[islot] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(smem_u32(&sh.info_full[islot]));
                }
                break;
            }
            const bool is_gu = it < n_gu;
            const DecArgs& P = is_gu ? gu : dn;
            const int id = is_gu ? it : it - n_gu;
            const int ti = id / P.row_blocks, rb = id % P.row_blocks;
            const int4 tile = P.tiles[ti];
            const int gu_target = gu.row_blocks + gu.dep.bias;
            if (!is_gu && lane == 0 && (int)ld_acquire(gu_done + ti) < gu_target) {
                const long long t0 = clock64();
                while ((int)ld_acquire(gu_done + ti) < gu_target) {
                    if (clock64() - t0 > gu.dep.limit) {
                        *abort = 1;
                        break;
                    }
                    __nanosleep(256);
                }
            }
            if (__shfl_sync(0xffffffffu, *abort, 0)) break;
            if (lane == 0) {
                sh.info[islot] = make_int4(it, tile.x, tile.y, tile.z);
                mbar_arrive(smem_u32(&sh.info_full[islot]));
            }
            // the item's rows: TMA rows, and this lane's scale row
            const int64_t ebase = (int64_t)tile.x * P.rows_per_expert;
            int64_t srow;
            if (is_gu) srow = ebase + (lane < 16 ? rb * 16 + lane : P.I + rb * 16 + (lane - 16));
            else srow = ebase + rb * 32 + lane;
            // scale bytes of the row: one per 32 elements (2-bit) or per 16 (NVFP4)
            const uint8_t* ssrc = P.scales + srow * (P.K / (kW4 ? 16 : 32));
            const int nch = P.K / kChunk;
            constexpr int rbytes = (int)F::kRowBytes;
            for (int ch = 0; ch < nch; ++ch, ++q) {
                const uint32_t slot = q % F::kSlots;
                if (lane == 0) ok = mbar_wait(smem_u32(&sh.empty[slot]), ((q / F::kSlots) & 1u) ^ 1u, abort);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                const uint32_t fb = smem_u32(&sh.full[slot]);
                const uint32_t dst = ring_addr + slot * F::kSlotBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, F::kSlotCodeBytes);
                    if (is_gu) {
                        tma_load_2d(dst, &gu_map, ch * rbytes, (int)(ebase + rb * 16), fb);
                        tma_load_2d(dst + 16 * rbytes, &gu_map, ch * rbytes, (int)(ebase + P.I + rb * 16), fb);
                    } else {
                        tma_load_2d(dst, &dn_map, ch * rbytes, (int)(ebase + rb * 32), fb);
                    }
                }
                if constexpr (kW4) cp_async16(dst + F::kSlotCodeBytes + lane * 16, ssrc + ch * 16);
                else cp_async8(dst + F::kSlotCodeBytes + lane * 8, ssrc + ch * 8);
                cp_async_arrive_noinc(fb);
            }
            if (!ok) break;
            int nxt = 0;
            if (lane == 0) nxt = atomicAdd(queue, 1);
            it = __shfl_sync(0xffffffffu, nxt, 0);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy of this warp outlives the CTA
    } else {
        // ------------------------------------------------ consumer warps
        const SelConst k = sel_const_regs();
        // AND of every lut word used: a valid scale's lut word has bit 31 set, an
        // invalid one is 0, so the AND is 0 exactly when a bad scale byte was read.
        uint32_t lut_and = 0xFFFFFFFFu;
        uint32_t qbase = 0;
        for (int n = 0;; ++n) {
            // one thread waits for the next item and decides whether to stop; the
            // barrier hands both to every consumer warp, so all four always take
            // the same path and meet at the same barriers
            const uint32_t islot = (uint32_t)n % kInfo;
            if (tid == 0) {
                const bool ok = mbar_wait(smem_u32(&sh.info_full[islot]), (uint32_t)(n / kInfo) & 1u, abort);
                sh.cur_info = ok ? sh.info[islot] : make_int4(-1, 0, 0, 0);
                sh.stop = !ok || *abort;
            }
            consumer_sync();
            const int4 info = sh.cur_info;
            if (sh.stop || info.x < 0) break;
            if (info.x < n_gu) {
                const int rb = info.x % gu.row_blocks;
                if (info.w <= 8) run_item<true, 1, kW4>(gu, k, sh, ring, qbase, info.z, info.w, rb, info.y, lut_and);
                else run_item<true, 2, kW4>(gu, k, sh, ring, qbase, info.z, info.w, rb, info.y, lut_and);
                qbase += (uint32_t)(gu.K / kChunk);
                // run_item ends with a consumer barrier after its h stores
                if (tid == 0) {
                    __threadfence();
                    atomicAdd(gu_done + info.x / gu.row_blocks, 1);
                }
            } else {
                const int rb = (info.x - n_gu) % dn.row_blocks;
                if (info.w <= 8) run_item<false, 1, kW4>(dn, k, sh, ring, qbase, info.z, info.w, rb, info.y, lut_and);
                else run_item<false, 2, kW4>(dn, k, sh, ring, qbase, info.z, info.w, rb, info.y, lut_and);
                qbase += (uint32_t)(dn.K / kChunk);
                // The last of the n_tiles items that wrote rows [32 rb, 32 rb + 32) of
                // the pair slots sums them into y (fixed j order per token).  run_item
                // ended with a consumer barrier after the stage stores, so one fence by
                // the counting thread releases all of them (fences are cumulative).
                if (tid == 0) {
                    __threadfence();
                    sh.last_flag = (atomicAdd(dn.counters + rb, 1) == n_tiles - 1);
                }
                consumer_sync();
                if (sh.last_flag) {
                    __threadfence();
                    for (int i = tid; i < dn.T * 32; i += kWarps * 32) {
                        const int t = i >> 5, m = rb * 32 + (i & 31);
                        float s = 0.f;
                        for (int j = 0; j < dn.k; ++j) {
                            const int ej = __ldg(dn.ids + t * dn.k + j);
                            if ((unsigned)ej < (unsigned)dn.E) s += __ldcg(dn.stage + (int64_t)(t * dn.k + j) * dn.H + m);
                        }
                        __nv_bfloat16 yb = __float2bfloat16_rn(s);
                        dn.y[(int64_t)t * dn.H + m] = *reinterpret_cast<uint16_t*>(&yb);
                    }
                    if (tid == 0) dn.counters[rb] = 0;
                }
                consumer_sync();
            }
            if (lane == 0) mbar_arrive(smem_u32(&sh.info_empty[islot]));
        }
        if (lut_and == 0) flag_status(gu.status, MOE_W2_DEV_BAD_SCALE);
    }
    if (tid == 0 && *abort) flag_status(gu.status, kDevPipelineTimeout);
}

template <bool kW4>
cudaError_t launch_decode_mma_fmt(const int32_t* ids, const float* weights, const LayerPlanes& w, int32_t T,
                                  int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                                  const PhaseEvents& ev)
{
    using F = Fmt<kW4>;
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    constexpr int kDyn = F::kRingBytes + 128;
    static bool ready[kMaxDevices];
    static int occ_of[kMaxDevices];
    int dev = 0;
    cudaError_t e0 = once_per_device(ready, dev, [&](int d) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<kW4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_mma_kernel<kW4>, kThreads, kDyn);
        if (e != cudaSuccess) return e;
        occ_of[d] = std::max(occ, 1);
        return cudaSuccess;
    });
    if (e0 != cudaSuccess) return e0;
    const int occ = occ_of[dev];
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
    gp.dep = dependency_wait();
    gp.scale_2 = w.w13_scale_2;
    gp.s2_stride = 2;

    DecArgs dp = gp;
    dp.codes = w.w2_codes;
    dp.scales = w.w2_scales;
    dp.K = I;
    dp.rows_per_expert = H;
    dp.row_blocks = H / 32;
    dp.act = ws.h;
    dp.scale_2 = w.w2_scale_2;
    dp.s2_stride = 1;
    int32_t* gu_done = ws.counters + H / 32;   // [tiles], zeroed by the permutation kernel
    int32_t* queue = gu_done + tiles;          // item queue, zeroed by the permutation kernel

    // code tiles: one chunk of a row (64 bytes of 2-bit codes or 128 bytes of
    // e2m1, 256 elements) x 16 rows (gate_up: gate and up halves separately) or
    // x 32 rows (down)
    constexpr int per_byte = kW4 ? 2 : 4;
    CUtensorMap gu_map, dn_map;
    cudaError_t e = make_tmap_2d(&gu_map, w.w13_codes, false, (int64_t)E * 2 * I, H / per_byte, F::kRowBytes, 16, 0);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_2d(&dn_map, w.w2_codes, false, (int64_t)E * H, I / per_byte, F::kRowBytes, 32, 0)) !=
        cudaSuccess)
        return e;

    // at most occupancy x SMs (all resident at once when the GPU is otherwise
    // idle), and no more than the larger phase has items
    const int64_t grid = std::min<int64_t>((int64_t)sm_count() * occ,
                                           tiles * std::max<int64_t>(gp.row_blocks, dp.row_blocks));
    if ((e = ev.record(1, s)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)kDyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may start before the permutation ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, decode_mma_kernel<kW4>, gu_map, dn_map, gp, dp, gu_done, queue)) != cudaSuccess)
        return e;
    return ev.record(2, s);   // the combine is inside the kernel: phase 3 is empty
}

}  // namespace

cudaError_t launch_decode_mma(const int32_t* ids, const float* weights, const LayerPlanes& w, int32_t T, int32_t k,
                              const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                              const PhaseEvents& ev)
{
    return w.w4 ? launch_decode_mma_fmt<true>(ids, weights, w, T, k, ws, y, status, s, ev)
                : launch_decode_mma_fmt<false>(ids, weights, w, T, k, ws, y, status, s, ev);
}

}  // namespace moe_w2
