// Prefill path (T > 64): grouped expert GEMMs on the 5th-generation tensor cores.
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": 2-bit codes expanded
// in the kernel and fed to block-scaled tensor-core MMAs; the prefill GEMM is
// load-issue-bound on SM120, which their fragment-major activation repack
// ("AFRAG", page "The v0.24.0 port", section "Our hooks") addressed.  Here the
// activation tiles arrive by TMA (no per-thread load issue at all) and the
// weight codes are expanded by four warps straight into the UMMA operand layout.
// Page "The v0.24.0 port", "Deterministic unpermute" bullet: each pair's output
// is placed in its own slot and the k slots of a token are summed in a fixed
// order (no atomics).
//
// Launch sequence: gather (x rows in expert order, T16 layout) -> gate_up GEMM
// with the SiLU(gate)*up epilogue -> down GEMM whose epilogue multiplies by the
// router weight and stores the pair's fp32 row in its slot -> combine.
//
// GEMM kernel (one template, two epilogues).  Work item = (tile of <= 256 pairs
// of one expert, block of 128 weight rows).  For gate_up the 128 A rows are 64
// gate rows interleaved with their 64 up rows (A row 2i = gate i, 2i+1 = up i),
// so each gate/up pair of accumulator rows sits in adjacent TMEM lanes of one
// warp.  D[128 x N] (fp32) lives in tensor memory: lanes = weight rows,
// columns = pairs; two such accumulators (all 512 columns) let the epilogue of
// one item run while the next item's main loop fills the other.
//   warps 0-3  expand the A tile (thread r = A row r) into the 128B-swizzled
//              smem layout, from raw codes in shared memory (scale bytes are
//              loaded per thread one superstage ahead)
//   warp 4     TMA producer of the B tiles (activations, 64 pair rows per copy)
//   warp 5     MMA issuer (one thread): 4 x tcgen05.mma (K = 16) per stage
//   warps 6-9  epilogue: TMEM lanes 32*(warp % 4) .. +31
//   warp 10    TMA producer of the raw code tiles: one superstage (4 stages,
//              64 code bytes per A row) at a time, two superstages ahead
//
// The FP4 layer (page "vLLM-Moet wiki", "The kernels" and "FP4 recovery":
// moe_w4_mm over the NVFP4 experts) is the same kernel with kW4: a superstage
// is 2 stages (64 bytes of e2m1 per A row, 128 elements), the scale bytes are
// e4m3 per 16 elements (8 per superstage, as for 2-bit), every 16-element
// block becomes bf16 pairs through fp4_word_bf16 with its scale in the table,
// and the epilogues multiply by the tensors' scale_2.
#include <algorithm>
#include <type_traits>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kBK = 64;                  // K per pipeline stage
constexpr int kStages = 4;
constexpr int kRowsA = 128;              // UMMA M
constexpr int kMaxN = 256;               // pairs per tile (UMMA N <= 256)
constexpr int kBRows = 64;               // pair rows per B TMA box
constexpr int kExpThreads = 128;
constexpr int kThreads = 352;
constexpr int kSuper = 4;                // stages per code superstage (256 K, 64 code bytes per row; FP4: 2)
constexpr int kCSlots = 2;               // code superstages in flight
constexpr uint32_t kABytes = kRowsA * 128;
constexpr uint32_t kBBytes = kMaxN * 128;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kCodeRowBytes = kSuper * 16;          // code bytes per A row per superstage
constexpr uint32_t kCodeBytes = kRowsA * kCodeRowBytes;   // one superstage of raw codes, 64B-swizzled rows
constexpr uint32_t kSmemBytes = kStages * kStageBytes + kCSlots * kCodeBytes + 1024;
constexpr uint32_t kTmemCols = 512;            // two accumulators of kMaxN columns

struct GemmParams {
    const uint8_t* codes;    // plane codes of this projection [E][rows_per_expert][K/4]
    const uint8_t* scales;   // [E][rows_per_expert][K/32]
    int32_t K;
    int32_t rows_per_expert;
    int32_t I;               // gate_up: index of the first up row
    int32_t H;               // down: y width (stage row length)
    int32_t row_blocks;      // items per tile
    const int4* tiles;
    const int32_t* tile_count;
    uint16_t* h_t16;         // gate_up output [P][I]
    float* stage;            // down output [P][H]
    const int32_t* sorted;
    const float* weights;
    uint32_t* status;
    const float* scale_2;    // FP4 layer: per-tensor scale_2 of expert e at e * s2_stride (+1: up)
    int32_t s2_stride;
};

__device__ __forceinline__ uint32_t word_i(const uint4& q, int i)
{
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// Row pointers of expansion thread r for item `it` (codes and scales of its A row).
template <bool kGateUp, bool kW4>
__device__ __forceinline__ void item_row(const GemmParams& p, int it, int r, const uint8_t*& rc, const uint8_t*& rs)
{
    const int4 tile = p.tiles[it / p.row_blocks];
    const int rb = it % p.row_blocks;
    int row;
    if (kGateUp) row = (r & 1 ? p.I : 0) + rb * 64 + (r >> 1);
    else row = rb * kRowsA + r;
    const int64_t grow = (int64_t)tile.x * p.rows_per_expert + row;
    rc = p.codes + grow * (p.K / (kW4 ? 2 : 4));
    rs = p.scales + grow * (p.K / (kW4 ? 16 : 32));
}

template <bool kGateUp, bool kW4>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_gemm_kernel(const __grid_constant__ CUtensorMap bmap,
                                                                      const __grid_constant__ CUtensorMap cmap,
                                                                      GemmParams p)
{
    constexpr int kSup = kW4 ? 2 : kSuper;   // stages per code superstage
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t dfull_bar[2];
    __shared__ __align__(8) uint64_t dempty_bar[2];
    __shared__ __align__(8) uint64_t cfull_bar[kCSlots];
    __shared__ __align__(8) uint64_t cempty_bar[kCSlots];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ std::conditional_t<kW4, uint4, uint2> lut_tab[256];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t smem_base = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int s = tid; s < 256; s += kThreads) {
        if constexpr (kW4) {
            lut_tab[s] = make_fp4_lut((uint32_t)s);
        } else {
            ScaleLut l = make_lut((uint32_t)s);
            lut_tab[s] = make_uint2(l.lut, l.lo);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), kExpThreads + 1);
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&dfull_bar[b]), 1);
            mbar_init(smem_u32(&dempty_bar[b]), kExpThreads);
        }
        for (int c = 0; c < kCSlots; ++c) {
            mbar_init(smem_u32(&cfull_bar[c]), 1);
            mbar_init(smem_u32(&cempty_bar[c]), kExpThreads);
        }
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_sh), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int* abort = &abort_flag;

    const int n_items = *p.tile_count * p.row_blocks;
    const int nk = p.K / kBK;
    // items of this CTA: blockIdx.x + n * gridDim.x, n = 0 .. my_items-1
    const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    const int n_super = (nk + kSup - 1) / kSup;   // code superstages per item
    const uint32_t code_base = smem_base + kStages * kStageBytes;

    if (warp < 4) {
        // ------------------------------------------------ expanders
        const int r = tid;   // A row
        const SelConst k = sel_const_regs();
        uint32_t lut_min = 0xFFFFFFFFu;
        // this thread's row inside the code tile: gate_up puts gate rows in the
        // first 64 rows of the tile and up rows in the next 64
        const int trow = kGateUp ? ((r & 1) * 64 + (r >> 1)) : r;
        const uint32_t trow_addr = (uint32_t)trow * kCodeRowBytes;
        const uint32_t swz = (uint32_t)((trow >> 1) & 3);   // 64-byte swizzle: chunk j at j ^ ((row / 2) % 4)
        // scale bytes of superstage su of item n (one 8-byte load: 4 stages x 2
        // UE8M0 bytes, or 2 stages x 4 e4m3 bytes)
        uint32_t nan_seen = 0;
        auto load_scales = [&](int n, int su, uint2& s0) {
            const int it = blockIdx.x + n * (int)gridDim.x;
            const uint8_t *rc, *rs;
            item_row<kGateUp, kW4>(p, it, r, rc, rs);
            s0 = __ldg(reinterpret_cast<const uint2*>(rs + su * 8));
            if (kW4) nan_seen |= e4m3_nan_bytes(s0.x) | e4m3_nan_bytes(s0.y);
        };
        int n = 0, su = 0;           // current (item, superstage)
        uint2 sa = make_uint2(0, 0);
        if (my_items > 0) load_scales(0, 0, sa);
        uint32_t g = 0, u = 0;       // stage and superstage counters of the whole stream
        bool ok = my_items > 0;
        while (ok) {
            // prefetch the next superstage's scale bytes
            int n2 = n, su2 = su + 1;
            if (su2 == n_super) {
                su2 = 0;
                ++n2;
            }
            uint2 na = make_uint2(0, 0);
            if (n2 < my_items) load_scales(n2, su2, na);

            const uint32_t cslot = u % kCSlots;
            if (!mbar_wait(smem_u32(&cfull_bar[cslot]), (u / kCSlots) & 1u, abort)) break;
            const uint32_t ctile = code_base + cslot * kCodeBytes + trow_addr;
            const int s_end = min(kSup, nk - su * kSup);
#pragma unroll
            for (int s = 0; s < kSup; ++s) {
                if (s >= s_end) break;
                const uint32_t slot = g % kStages, ph = (g / kStages) & 1u;
                if constexpr (kW4) {
                    // 32 bytes of e2m1 (64 elements: four blocks of 16) and their four e4m3 bytes
                    const uint4 c0q = lds_u4(ctile + ((((uint32_t)(2 * s)) ^ swz) << 4));
                    const uint4 c1q = lds_u4(ctile + ((((uint32_t)(2 * s + 1)) ^ swz) << 4));
                    const uint32_t sw = s ? sa.y : sa.x;
                    if (!mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_tile = smem_base + slot * kStageBytes;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4& cq = i < 2 ? c0q : c1q;
                        const uint4 L = lut_tab[(sw >> (8 * i)) & 0xFFu];
                        uint32_t lo[4], hi[4];   // elements 0..7 and 8..15 of block i
                        fp4_word_bf16(word_i(cq, 2 * (i & 1)), L, lo[0], lo[1], lo[2], lo[3]);
                        fp4_word_bf16(word_i(cq, 2 * (i & 1) + 1), L, hi[0], hi[1], hi[2], hi[3]);
                        // T16 storage order of the block: (e0,e4)(e8,e12)(e1,e5)(e9,e13) | (e2,e6)(e10,e14)(e3,e7)(e11,e15)
                        sts_u4(a_tile + sw128_offset(r, 2 * i), make_uint4(lo[0], hi[0], lo[1], hi[1]));
                        sts_u4(a_tile + sw128_offset(r, 2 * i + 1), make_uint4(lo[2], hi[2], lo[3], hi[3]));
                    }
                } else {
                const uint4 cq = lds_u4(ctile + ((((uint32_t)s) ^ swz) << 4));
                const uint32_t cs = ((s & 2 ? sa.y : sa.x) >> (16 * (s & 1))) & 0xFFFFu;
                if (!mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1u, abort)) {
                    ok = false;
                    break;
                }
                const uint2 L0 = lut_tab[cs & 0xFF], L1 = lut_tab[cs >> 8];
                lut_min = min(lut_min, min(L0.x, L1.x));
                const uint32_t a_tile = smem_base + slot * kStageBytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint2 L = (i < 2) ? L0 : L1;
                    uint32_t lo[4], hi[4];
                    selectors(word_masks(word_i(cq, i), k), k, lo, hi);
                    uint4 c0, c1;
                    c0.x = prmt(L.x, L.y, lo[0]);
                    c0.y = prmt(L.x, L.y, hi[0]);
                    c0.z = prmt(L.x, L.y, lo[1]);
                    c0.w = prmt(L.x, L.y, hi[1]);
                    c1.x = prmt(L.x, L.y, lo[2]);
                    c1.y = prmt(L.x, L.y, hi[2]);
                    c1.z = prmt(L.x, L.y, lo[3]);
                    c1.w = prmt(L.x, L.y, hi[3]);
                    sts_u4(a_tile + sw128_offset(r, 2 * i), c0);
                    sts_u4(a_tile + sw128_offset(r, 2 * i + 1), c1);
                }
                }   // 2-bit planes
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full_bar[slot]));
                ++g;
            }
            if (!ok) break;
            mbar_arrive(smem_u32(&cempty_bar[cslot]));   // this thread is done reading the code tile
            ++u;
            n = n2;
            su = su2;
            sa = na;
            if (n >= my_items) break;
        }
        if (lut_min == 0 || nan_seen != 0) flag_status(p.status, MOE_W2_DEV_BAD_SCALE);
    } else if (warp == 4) {
        // ------------------------------------------------ TMA producer (B tiles)
        if (lane == 0) {
            prefetch_tmap(&bmap);
            uint32_t g = 0;
            for (int n = 0; n < my_items && !*abort; ++n) {
                const int it = blockIdx.x + n * (int)gridDim.x;
                const int4 tile = p.tiles[it / p.row_blocks];
                // boxes of kBRows pair rows; rows past the tile's pairs are loaded
                // too (the MMA reads only the first npad) or zero-filled past P
                const int q0 = tile.y, nbox = (tile.z + kBRows - 1) / kBRows;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t slot = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&empty_bar[slot]), ph ^ 1u, abort)) break;
                    const uint32_t fb = smem_u32(&full_bar[slot]);
                    mbar_arrive_expect_tx(fb, (uint32_t)nbox * kBRows * 128u);
                    const uint32_t b_tile = smem_base + slot * kStageBytes + kABytes;
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(b_tile + j * kBRows * 128u, &bmap, kk * kBK, q0 + kBRows * j, fb);
                    ++g;
                }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0;
            for (int n = 0; n < my_items && !*abort; ++n) {
                const int it = blockIdx.x + n * (int)gridDim.x;
                const int4 tile = p.tiles[it / p.row_blocks];
                const uint32_t npad = (tile.z + 15) & ~15;
                const uint32_t idesc = idesc_bf16_f32(kRowsA, npad);
                const uint32_t b = n & 1;
                // accumulator b is free once the epilogue of item n-2 drained it
                if (!mbar_wait(smem_u32(&dempty_bar[b]), ((n >> 1) & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                const uint32_t acc = tmem + b * kMaxN;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t slot = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(smem_u32(&full_bar[slot]), ph, abort)) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_base + slot * kStageBytes;
                    const uint64_t ad = smem_desc_sw128(a_addr), bd = smem_desc_sw128(a_addr + kABytes);
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        umma_f16_ss(acc, ad + 2 * k4, bd + 2 * k4, idesc, (kk | k4) != 0);
                    umma_commit(smem_u32(&empty_bar[slot]));
                    ++g;
                }
                umma_commit(smem_u32(&dfull_bar[b]));
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------ TMA producer (raw code tiles)
        if (lane == 0) {
            prefetch_tmap(&cmap);
            uint32_t u = 0;
            for (int n = 0; n < my_items && !*abort; ++n) {
                const int it = blockIdx.x + n * (int)gridDim.x;
                const int4 tile = p.tiles[it / p.row_blocks];
                const int rb = it % p.row_blocks;
                const int64_t ebase = (int64_t)tile.x * p.rows_per_expert;
                for (int su = 0; su < n_super; ++su) {
                    const uint32_t cslot = u % kCSlots;
                    if (!mbar_wait(smem_u32(&cempty_bar[cslot]), ((u / kCSlots) & 1u) ^ 1u, abort)) break;
                    const uint32_t fb = smem_u32(&cfull_bar[cslot]);
                    mbar_arrive_expect_tx(fb, kCodeBytes);
                    const uint32_t dst = code_base + cslot * kCodeBytes;
                    const int x = su * (int)kCodeRowBytes;   // byte column of the superstage (64 bytes either way)
                    if (kGateUp) {
                        tma_load_2d(dst, &cmap, x, (int)(ebase + rb * 64), fb);
                        tma_load_2d(dst + 64 * kCodeRowBytes, &cmap, x, (int)(ebase + p.I + rb * 64), fb);
                    } else {
                        tma_load_2d(dst, &cmap, x, (int)(ebase + rb * kRowsA), fb);
                    }
                    ++u;
                }
            }
        }
    } else {
        // ------------------------------------------------ epilogue (warps 6-9)
        const int quarter = warp & 3;           // TMEM lanes 32*quarter .. +31
        const int r = 32 * quarter + lane;      // A row
        for (int n = 0; n < my_items && !*abort; ++n) {
            const int it = blockIdx.x + n * (int)gridDim.x;
            const int4 tile = p.tiles[it / p.row_blocks];
            const int rb = it % p.row_blocks;
            const int q0 = tile.y, nrows = tile.z;
            const uint32_t b = n & 1;
            // FP4 layer: this row's tensor scale_2 (gate_up: gate rows even, up rows odd)
            const float s2 = kW4 ? __ldg(p.scale_2 + (int64_t)tile.x * p.s2_stride + (kGateUp ? (r & 1) : 0)) : 1.f;
            if (!mbar_wait(smem_u32(&dfull_bar[b]), (n >> 1) & 1u, abort)) break;
            tc_fence_after();
            const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + b * kMaxN;
            for (int c0 = 0; c0 < nrows; c0 += 32) {
                float v[32];
                tmem_ld32(lane_base + c0, v);
                if (kW4) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= s2;
                }
                if (kGateUp) {
                    const int nn = rb * 64 + (r >> 1);
                    const int pos = t16_pos(nn);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float up = __shfl_down_sync(0xffffffffu, v[j], 1);
                        if (!(r & 1) && c0 + j < nrows) {
                            __nv_bfloat16 hb = __float2bfloat16_rn(silu_f(v[j]) * up);
                            p.h_t16[(int64_t)(q0 + c0 + j) * p.I + pos] = *reinterpret_cast<uint16_t*>(&hb);
                        }
                    }
                } else {
                    // lane j fetches column c0+j's pair id and router weight once;
                    // shuffles hand them to every lane
                    const int m = rb * kRowsA + r;
                    int my_pr = 0;
                    float my_w = 0.f;
                    if (c0 + lane < nrows) {
                        my_pr = __ldg(p.sorted + q0 + c0 + lane);
                        my_w = __ldg(p.weights + my_pr);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int pr = __shfl_sync(0xffffffffu, my_pr, j);
                        const float wt = __shfl_sync(0xffffffffu, my_w, j);
                        if (c0 + j < nrows) p.stage[(int64_t)pr * p.H + m] = wt * v[j];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&dempty_bar[b]));
        }
    }

    tc_fence_before();
    cta_barrier_all_threads();   // every thread done before tensor memory is freed
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && abort_flag) flag_status(p.status, kDevPipelineTimeout);
}

template <bool kW4>
cudaError_t launch_prefill_fmt(const uint16_t* x, const int32_t* ids, const float* weights, const LayerPlanes& w,
                               int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status,
                               cudaStream_t s, const PhaseEvents& ev)
{
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    static bool ready[kMaxDevices];
    int dev = 0;
    cudaError_t e0 = once_per_device(ready, dev, [](int) {
        cudaError_t e = cudaFuncSetAttribute(tc_expert_gemm_kernel<true, kW4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        return cudaFuncSetAttribute(tc_expert_gemm_kernel<false, kW4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
    });
    if (e0 != cudaSuccess) return e0;
    const int sms = sm_count();

    cudaError_t e = launch_gather(x, ws.sorted, ws.offsets, E, k, H, P, ws.xa, s);
    if (e != cudaSuccess) return e;

    CUtensorMap xmap, hmap, c13map, c2map;
    if ((e = make_tmap_2d(&xmap, ws.xa, true, P, H, 64, kBRows, 128)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&hmap, ws.h, true, P, I, 64, kBRows, 128)) != cudaSuccess) return e;
    // raw code tiles: 64 bytes (256 2-bit codes or 128 e2m1) x 64 rows (gate_up:
    // gate and up halves) or 128 rows
    constexpr int per_byte = kW4 ? 2 : 4;
    if ((e = make_tmap_2d(&c13map, w.w13_codes, false, (int64_t)E * 2 * I, H / per_byte, kCodeRowBytes, 64, 64)) !=
        cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&c2map, w.w2_codes, false, (int64_t)E * H, I / per_byte, kCodeRowBytes, kRowsA, 64)) !=
        cudaSuccess)
        return e;

    if ((e = ev.record(1, s)) != cudaSuccess) return e;
    GemmParams gp{};
    gp.codes = w.w13_codes;
    gp.scales = w.w13_scales;
    gp.K = H;
    gp.rows_per_expert = 2 * I;
    gp.I = I;
    gp.H = H;
    gp.row_blocks = I / 64;
    gp.tiles = ws.tiles;
    gp.tile_count = ws.tile_count;
    gp.h_t16 = ws.h;
    gp.stage = ws.stage;
    gp.sorted = ws.sorted;
    gp.weights = weights;
    gp.status = status;
    gp.scale_2 = w.w13_scale_2;
    gp.s2_stride = 2;
    const int64_t max_items = max_tiles(P, E, false) * (I / 64);
    tc_expert_gemm_kernel<true, kW4><<<(int)std::min<int64_t>(sms, max_items), kThreads, kSmemBytes, s>>>(xmap, c13map,
                                                                                                        gp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    if ((e = ev.record(2, s)) != cudaSuccess) return e;
    GemmParams dp = gp;
    dp.codes = w.w2_codes;
    dp.scales = w.w2_scales;
    dp.K = I;
    dp.rows_per_expert = H;
    dp.row_blocks = H / kRowsA;
    dp.scale_2 = w.w2_scale_2;
    dp.s2_stride = 1;
    const int64_t max_items_d = max_tiles(P, E, false) * (H / kRowsA);
    tc_expert_gemm_kernel<false, kW4><<<(int)std::min<int64_t>(sms, max_items_d), kThreads, kSmemBytes, s>>>(
        hmap, c2map, dp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    return launch_combine(ws.stage, ids, T, k, E, H, 1, 0, false, y, s);
}

}  // namespace

cudaError_t launch_prefill(const uint16_t* x, const int32_t* ids, const float* weights, const LayerPlanes& w,
                           int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                           const PhaseEvents& ev)
{
    return w.w4 ? launch_prefill_fmt<true>(x, ids, weights, w, T, k, ws, y, status, s, ev)
                : launch_prefill_fmt<false>(x, ids, weights, w, T, k, ws, y, status, s, ev);
}

}  // namespace moe_w2
