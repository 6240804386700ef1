// Decode path (T <= 64): the 2-bit planes of every active expert are streamed
// from HBM once per layer; tensor cores do the dot products.
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": codes expanded in
// registers through a byte-permute lookup table and fed to tensor-core MMAs;
// section "FP4 recovery": decode is HBM-bound, the 2-bit read is the cost.  Page
// "The v0.24.0 port", section "Benchmarks": tokens grouped by expert, so each
// active expert's weights are read once per step however many tokens use it.
//
// GB300 design.  The legacy mma.sync path is far too slow on sm_103 for a GEMV
// that wastes most of N, and expanding the weights into shared memory would need
// ~2 bytes of st.shared per code at HBM rate.  So the expanded A operand goes to
// tensor memory instead:
//   TMA        one producer thread streams 128-row x 128-code tiles of the packed
//              codes into a deep shared ring (12 stages, 48 KB per CTA, released
//              by the expanders once a tile is in TMEM);
//              another streams the pairs' activation rows (expert order, T16
//              layout) into 128B-swizzled B tiles;
//   expanders  two warpgroups, alternating stages; thread r owns A row r: it
//              reads its 32 code bytes, expands them with one byte-permute per
//              weight pair (scale folded into a per-block table) and writes the
//              64 bf16 pairs into its TMEM lane with tcgen05.st;
//   MMA        one thread issues tcgen05.mma (A from TMEM, B from shared memory,
//              D in TMEM): 8 x (M=128, N=pairs padded to 16, K=16) per stage;
//   epilogue   the expanders read D back: SiLU(gate)*up -> h (gate_up), or
//              router weight * D -> the pair's fp32 slot (down); a small
//              combine kernel then sums each token's k slots in a fixed order.
// Work item = (tile of <= 64 pairs of one expert, 128 weight rows).  For gate_up
// the A rows interleave gate and up rows (A row 2i = gate i, 2i+1 = up i).
#include <algorithm>
#include <mutex>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kKS = 128;                  // K per stage
constexpr int kSC = 12;                   // code-tile ring (HBM latency cover: 48 KB per CTA)
constexpr int kSB = 3;                    // activation-tile ring (L2-resident rows)
constexpr int kSA = 3;                    // TMEM A ring
constexpr int kMaxN = 64;                 // pairs per decode tile
constexpr int kGroups = 2;                // expander warpgroups
constexpr int kThreads = kGroups * 128 + 96;   // + code producer, B producer, MMA issuer
constexpr uint32_t kCodeBytes = 128 * 32;          // 128 rows x 32 code bytes
constexpr uint32_t kBAtom = kMaxN * 128;           // 64 bf16 of K for kMaxN rows
constexpr uint32_t kBBytes = 2 * kBAtom;           // K = 128: two 128-byte atoms
constexpr uint32_t kSmemBytes = kSC * kCodeBytes + kSB * kBBytes + 1024;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kDCol = 0;                      // D: columns [0, 64)
constexpr uint32_t kACol = 64;                     // A ring: 3 x 64 columns

struct DecodeParams {
    int32_t K;
    int32_t rows_per_expert;   // 2I or H
    int32_t I;
    int32_t H;
    int32_t k;                 // top_k (pair -> token)
    int32_t row_blocks;
    const uint8_t* scales;     // [E][rows_per_expert][K/32]
    const int4* tiles;
    const int32_t* tile_count;
    const int32_t* sorted;
    const float* weights;
    uint16_t* h_t16;           // gate_up output [P][I]
    float* stage;              // down output [P][H]
    uint32_t* status;
};

__device__ __forceinline__ uint32_t word_of(const uint4& q, int i)
{
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// Expand one 16-code word into 8 bf16 pairs in T16 storage order.
__device__ __forceinline__ void expand_word(uint32_t w, const ScaleLut& L, uint32_t* o)
{
    const uint32_t s0 = code_selector<0>(w), s1 = code_selector<1>(w);
    const uint32_t s2 = code_selector<2>(w), s3 = code_selector<3>(w);
    o[0] = expand_pair(L, s0);
    o[1] = expand_pair(L, s0 >> 16);
    o[2] = expand_pair(L, s1);
    o[3] = expand_pair(L, s1 >> 16);
    o[4] = expand_pair(L, s2);
    o[5] = expand_pair(L, s2 >> 16);
    o[6] = expand_pair(L, s3);
    o[7] = expand_pair(L, s3 >> 16);
}

template <bool kGateUp>
__global__ void __launch_bounds__(kThreads, 2) tc_decode_kernel(const __grid_constant__ CUtensorMap cmap,
                                                             const __grid_constant__ CUtensorMap bmap,
                                                             DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t cfull_bar[kSC];    // code tile landed (TMA bytes)
    __shared__ __align__(8) uint64_t cempty_bar[kSC];   // code tile consumed by its expander group (128)
    __shared__ __align__(8) uint64_t bfull_bar[kSB];    // activation tile landed (TMA bytes)
    __shared__ __align__(8) uint64_t bempty_bar[kSB];   // MMAs reading it done (commit)
    __shared__ __align__(8) uint64_t afull_bar[kSA];    // expanded A in TMEM (128)
    __shared__ __align__(8) uint64_t aempty_bar[kSA];   // MMAs reading it done (commit)
    __shared__ __align__(8) uint64_t dfull_bar;         // accumulator complete (commit)
    __shared__ __align__(8) uint64_t dempty_bar;        // epilogue done reading D (256)
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ uint2 lut_tab[256];

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* b_ring = smem;                           // kSB x 16 KB (1 KB aligned)
    uint8_t* code_ring = smem + kSB * kBBytes;        // kSC x 4 KB
    const uint32_t code_ring_s = smem_u32(code_ring), b_ring_s = smem_u32(b_ring);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    for (int s = tid; s < 256; s += kThreads) {
        ScaleLut l = make_lut((uint32_t)s);
        lut_tab[s] = make_uint2(l.lut, l.lo);
    }
    if (tid == 0) {
        for (int s = 0; s < kSC; ++s) {
            mbar_init(smem_u32(&cfull_bar[s]), 1);
            mbar_init(smem_u32(&cempty_bar[s]), 128);
        }
        for (int s = 0; s < kSB; ++s) {
            mbar_init(smem_u32(&bfull_bar[s]), 1);
            mbar_init(smem_u32(&bempty_bar[s]), 1);
        }
        for (int s = 0; s < kSA; ++s) {
            mbar_init(smem_u32(&afull_bar[s]), 128);
            mbar_init(smem_u32(&aempty_bar[s]), 1);
        }
        mbar_init(smem_u32(&dfull_bar), 1);
        mbar_init(smem_u32(&dempty_bar), kGroups * 128);
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
    const int nk = p.K / kKS;

    if (warp < kGroups * 4) {
        // ------------------------------------------------ expanders + epilogue
        const int grp = warp >> 2, r = tid & 127, wq = warp & 3;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
        // A row r sits in code-tile row crow; its two 16-byte chunks are read in
        // the order (sw, sw^1) so 8 consecutive threads touch 8 distinct banks.
        const int crow = kGateUp ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
        const int sw = kGateUp ? (r & 1) : ((r >> 2) & 1);
        uint32_t g = 0, items_done = 0, lut_min = 0xFFFFFFFFu;
        for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
            const int4 tile = p.tiles[it / p.row_blocks];
            const int rb = it % p.row_blocks;
            const int e = tile.x, q0 = tile.y, nrows = tile.z;
            const int row = kGateUp ? ((r & 1 ? p.I : 0) + rb * 64 + (r >> 1)) : rb * 128 + r;
            const uint32_t* rs =
                reinterpret_cast<const uint32_t*>(p.scales + ((int64_t)e * p.rows_per_expert + row) * (p.K / 32));
            // stage gs = g + kk belongs to group gs % kGroups
            const int kk0 = (int)(((uint32_t)grp + kGroups - (g % kGroups)) % kGroups);
            uint32_t sq[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) sq[u] = (kk0 + kGroups * u < nk) ? __ldg(rs + kk0 + kGroups * u) : 0u;

            bool ok = true;
            for (int kb = kk0; kb < nk && ok; kb += 4 * kGroups) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int kk = kb + kGroups * u;
                    if (kk >= nk) break;
                    const uint32_t sc = sq[u];
                    sq[u] = (kk + 4 * kGroups < nk) ? __ldg(rs + kk + 4 * kGroups) : 0u;
                    const uint32_t gs = g + kk;
                    const uint32_t cs = gs % kSC, cph = (gs / kSC) & 1u;
                    const uint32_t as = gs % kSA, aph = (gs / kSA) & 1u;
                    if (!mbar_wait(smem_u32(&cfull_bar[cs]), cph, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t ct = code_ring_s + cs * kCodeBytes + crow * 32;
                    const uint4 f = lds_u4(ct + 16 * sw);
                    const uint4 s2 = lds_u4(ct + 16 * (sw ^ 1));
                    const uint4 ch0 = sw ? s2 : f, ch1 = sw ? f : s2;
                    const uint2 t0 = lut_tab[sc & 0xFF], t1 = lut_tab[(sc >> 8) & 0xFF];
                    const uint2 t2 = lut_tab[(sc >> 16) & 0xFF], t3 = lut_tab[sc >> 24];
                    lut_min = min(lut_min, min(min(t0.x, t1.x), min(t2.x, t3.x)));
                    if (!mbar_wait(smem_u32(&aempty_bar[as]), aph ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t regs[32];
                    expand_word(ch0.x, ScaleLut{t0.x, t0.y}, regs + 0);
                    expand_word(ch0.y, ScaleLut{t0.x, t0.y}, regs + 8);
                    expand_word(ch0.z, ScaleLut{t1.x, t1.y}, regs + 16);
                    expand_word(ch0.w, ScaleLut{t1.x, t1.y}, regs + 24);
                    const uint32_t acol = lane_addr + kACol + as * 64;
                    tmem_st32_sync(acol, regs);
                    expand_word(ch1.x, ScaleLut{t2.x, t2.y}, regs + 0);
                    expand_word(ch1.y, ScaleLut{t2.x, t2.y}, regs + 8);
                    expand_word(ch1.z, ScaleLut{t3.x, t3.y}, regs + 16);
                    expand_word(ch1.w, ScaleLut{t3.x, t3.y}, regs + 24);
                    tmem_st32_sync(acol + 32, regs);
                    tc_fence_before();
                    mbar_arrive(smem_u32(&afull_bar[as]));
                    // Release the code tile only once its bytes are in TMEM.  Releasing
                    // right after the shared loads let the next TMA fill of the slot
                    // corrupt rows that were still being read (seen at T=32 with two
                    // CTAs per SM); this ordering was verified race-free.
                    mbar_arrive(smem_u32(&cempty_bar[cs]));
                }
            }
            g += nk;
            if (!ok || *abort) break;

            // epilogue: this group's 32 accumulator columns (pairs c0 .. c0+31)
            if (!mbar_wait(smem_u32(&dfull_bar), items_done & 1u, abort)) break;
            ++items_done;
            tc_fence_after();
            for (int c0 = 32 * grp; c0 < nrows; c0 += 32 * kGroups) {
                float v[32];
                tmem_ld32(lane_addr + kDCol + c0, v);
                if (kGateUp) {
                    const int pos = t16_pos(rb * 64 + (r >> 1));
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float up = __shfl_down_sync(0xffffffffu, v[j], 1);
                        if (!(r & 1) && c0 + j < nrows) {
                            __nv_bfloat16 hb = __float2bfloat16_rn(silu_f(v[j]) * up);
                            p.h_t16[(int64_t)(q0 + c0 + j) * p.I + pos] = *reinterpret_cast<uint16_t*>(&hb);
                        }
                    }
                } else {
                    const int m = rb * 128 + r;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (c0 + j < nrows) {
                            const int pr = __ldg(p.sorted + q0 + c0 + j);
                            p.stage[(int64_t)pr * p.H + m] = __ldg(p.weights + pr) * v[j];
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&dempty_bar));
        }
        if (lut_min == 0) flag_status(p.status, MOE_W2_DEV_BAD_SCALE);
    } else if (warp == kGroups * 4) {
        // ------------------------------------------------ code-tile producer (TMA)
        if (lane == 0) {
            prefetch_tmap(&cmap);
            uint32_t g = 0;
            for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
                const int4 tile = p.tiles[it / p.row_blocks];
                const int rb = it % p.row_blocks;
                const int e = tile.x;
                const int rowA = kGateUp ? e * p.rows_per_expert + rb * 64 : e * p.rows_per_expert + rb * 128;
                const int rowB = kGateUp ? rowA + p.I : rowA + 64;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t gs = g + kk, cs = gs % kSC, ph = (gs / kSC) & 1u;
                    if (!mbar_wait(smem_u32(&cempty_bar[cs]), ph ^ 1u, abort)) break;
                    const uint32_t fb = smem_u32(&cfull_bar[cs]);
                    mbar_arrive_expect_tx(fb, kCodeBytes);
                    const uint32_t cdst = code_ring_s + cs * kCodeBytes;
                    tma_load_2d(cdst, &cmap, kk * 32, rowA, fb);
                    tma_load_2d(cdst + 64 * 32, &cmap, kk * 32, rowB, fb);
                }
                g += nk;
            }
        }
    } else if (warp == kGroups * 4 + 1) {
        // ------------------------------------------------ activation-tile producer (TMA)
        if (lane == 0) {
            prefetch_tmap(&bmap);
            uint32_t g = 0;
            for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
                const int4 tile = p.tiles[it / p.row_blocks];
                const int q0 = tile.y, npad = (tile.z + 15) & ~15;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t gs = g + kk, bs = gs % kSB, ph = (gs / kSB) & 1u;
                    if (!mbar_wait(smem_u32(&bempty_bar[bs]), ph ^ 1u, abort)) break;
                    const uint32_t fb = smem_u32(&bfull_bar[bs]);
                    mbar_arrive_expect_tx(fb, (uint32_t)npad * 256u);
                    const uint32_t bdst = b_ring_s + bs * kBBytes;
                    for (int a = 0; a < 2; ++a)
                        for (int j = 0; j < npad / 16; ++j)
                            tma_load_2d(bdst + a * kBAtom + j * 2048u, &bmap, kk * kKS + a * 64, q0 + 16 * j, fb);
                }
                g += nk;
            }
        }
    } else {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0, items = 0;
            for (int it = blockIdx.x; it < n_items && !*abort; it += gridDim.x) {
                const int4 tile = p.tiles[it / p.row_blocks];
                const uint32_t npad = (tile.z + 15) & ~15;
                const uint32_t idesc = idesc_bf16_f32(128, npad);
                if (!mbar_wait(smem_u32(&dempty_bar), (items & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t gs = g + kk;
                    const uint32_t as = gs % kSA, aph = (gs / kSA) & 1u;
                    const uint32_t bs = gs % kSB, bph = (gs / kSB) & 1u;
                    if (!mbar_wait(smem_u32(&afull_bar[as]), aph, abort) ||
                        !mbar_wait(smem_u32(&bfull_bar[bs]), bph, abort))
                        break;
                    tc_fence_after();
                    const uint32_t a_t = tmem + kACol + as * 64;
                    const uint32_t b_s = b_ring_s + bs * kBBytes;
#pragma unroll
                    for (int k16 = 0; k16 < 8; ++k16)
                        umma_f16_ts(tmem + kDCol, a_t + 8 * k16,
                                    smem_desc_sw128(b_s + (k16 >> 2) * kBAtom) + 2 * (k16 & 3), idesc,
                                    (kk | k16) != 0);
                    umma_commit(smem_u32(&aempty_bar[as]));
                    umma_commit(smem_u32(&bempty_bar[bs]));
                }
                umma_commit(smem_u32(&dfull_bar));
                ++items;
                g += nk;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && abort_flag) flag_status(p.status, kDevPipelineTimeout);
}

}  // namespace

cudaError_t launch_decode(const uint16_t* x, const int32_t* ids, const float* weights, const moe_w2_planes& w,
                          int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                          const PhaseEvents& ev)
{
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    // 100 KB of dynamic shared memory keeps it at two CTAs per SM (2 x 256 TMEM columns)
    constexpr int kDynSmem = 100 * 1024;
    static_assert(kSmemBytes <= kDynSmem, "shared-memory budget");
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(tc_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kDynSmem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tc_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int sms = sm_count();
    cudaError_t e = launch_gather(x, ws.sorted, ws.offsets, E, k, H, P, ws.xa, s);
    if (e != cudaSuccess) return e;

    CUtensorMap c13, c2, xmap, hmap;
    if ((e = make_tmap_2d(&c13, w.w13_codes, false, (int64_t)E * 2 * I, H / 4, 32, 64, false)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&c2, w.w2_codes, false, (int64_t)E * H, I / 4, 32, 64, false)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&xmap, ws.xa, true, P, H, 64, 16, true)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&hmap, ws.h, true, P, I, 64, 16, true)) != cudaSuccess) return e;

    DecodeParams gp{};
    gp.K = H;
    gp.rows_per_expert = 2 * I;
    gp.I = I;
    gp.H = H;
    gp.k = k;
    gp.row_blocks = I / 64;
    gp.scales = w.w13_scales;
    gp.tiles = ws.tiles;
    gp.tile_count = ws.tile_count;
    gp.sorted = ws.sorted;
    gp.weights = weights;
    gp.h_t16 = ws.h;
    gp.stage = ws.stage;
    gp.status = status;
    const int64_t tiles = max_tiles(P, E, true);
    if ((e = ev.record(1, s)) != cudaSuccess) return e;
    tc_decode_kernel<true><<<(int)std::min<int64_t>(tiles * (I / 64), 2 * (int64_t)sms), kThreads, kDynSmem, s>>>(
        c13, xmap, gp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    DecodeParams dp = gp;
    dp.K = I;
    dp.rows_per_expert = H;
    dp.row_blocks = H / 128;
    dp.scales = w.w2_scales;
    if ((e = ev.record(2, s)) != cudaSuccess) return e;
    tc_decode_kernel<false><<<(int)std::min<int64_t>(tiles * (H / 128), 2 * (int64_t)sms), kThreads, kDynSmem, s>>>(
        c2, hmap, dp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    (void)ids;
    return launch_combine(ws.stage, ids, T, k, E, H, y, s);
}

}  // namespace moe_w2
