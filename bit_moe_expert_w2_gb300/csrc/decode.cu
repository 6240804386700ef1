// Decode path (few tokens): the 2-bit planes of every active expert are
// streamed from HBM exactly once per layer and expanded in registers.
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": in-register decode of
// the codes through a byte-permute lookup table feeding tensor-core MMAs;
// section "FP4 recovery": decode is HBM-bound, so the 2-bit read is the cost.
// Page "The v0.24.0 port", section "Benchmarks": the per-step expert working set
// grows sublinearly with batch, because tokens are grouped by expert.
//
// Code expansion: one byte-permute per pair of weights; its table (four high
// bytes of the bf16 values +-1, +-4 times the block's power-of-two scale, and the
// shared low byte) comes from a 256-entry shared-memory table indexed by the
// UE8M0 byte.  Dot products run on mma.sync m16n8k16 (bf16 in, fp32 accumulate):
// A = 16 weight rows expanded in registers, B = up to 8 tokens/pairs whose
// activations sit in T16 order so every B fragment is one 64-bit load.
//
// Per 256-wide K chunk a row is 64 code bytes; thread c of a quad owns bytes
// [16c, 16c+16), i.e. four 16-code words; MMA (word i, r) takes codes (r, r+4)
// and (r+8, r+12) of word i from every thread of the quad.
#include <algorithm>

#include "common.cuh"

namespace moe_w2 {

namespace {

constexpr int kChunk = 256;   // K elements per chunk
constexpr int kNT = 4;        // n-tiles of 8 pairs per pass
constexpr int kPairsPerPass = 8 * kNT;

__device__ __forceinline__ void init_lut_table(uint2* tab)
{
    for (int s = threadIdx.x; s < 256; s += blockDim.x) {
        ScaleLut l = make_lut((uint32_t)s);
        tab[s] = make_uint2(l.lut, l.lo);
    }
}

__device__ __forceinline__ uint32_t word_of(const uint4& q, int i)
{
    return i == 0 ? q.x : i == 1 ? q.y : i == 2 ? q.z : q.w;
}

// One 256-wide K chunk: rows ra (A rows g) and rb (A rows g+8), the thread's 16
// code bytes of each and their two block luts; B rows per n-tile.
template <int NT>
__device__ __forceinline__ void chunk_mma(float (&d)[NT][4], const uint4& qa, const uint4& qb, const uint2& la0,
                                          const uint2& la1, const uint2& lb0, const uint2& lb1,
                                          const uint16_t* const (&brow)[NT], const bool (&bval)[NT], int nt_used,
                                          int boff)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wa = word_of(qa, i), wb = word_of(qb, i);
        const ScaleLut LA = (i < 2) ? ScaleLut{la0.x, la0.y} : ScaleLut{la1.x, la1.y};
        const ScaleLut LB = (i < 2) ? ScaleLut{lb0.x, lb0.y} : ScaleLut{lb1.x, lb1.y};
        uint4 B0[NT], B1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            B0[nt] = make_uint4(0, 0, 0, 0);
            B1[nt] = make_uint4(0, 0, 0, 0);
            if (nt < nt_used && bval[nt]) {
                B0[nt] = ldg_u4(brow[nt] + boff + i * 16);
                B1[nt] = ldg_u4(brow[nt] + boff + i * 16 + 8);
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const uint32_t sa = (r == 0) ? code_selector<0>(wa) : (r == 1) ? code_selector<1>(wa)
                              : (r == 2) ? code_selector<2>(wa) : code_selector<3>(wa);
            const uint32_t sb = (r == 0) ? code_selector<0>(wb) : (r == 1) ? code_selector<1>(wb)
                              : (r == 2) ? code_selector<2>(wb) : code_selector<3>(wb);
            uint32_t a[4];
            a[0] = expand_pair(LA, sa);
            a[1] = expand_pair(LB, sb);
            a[2] = expand_pair(LA, sa >> 16);
            a[3] = expand_pair(LB, sb >> 16);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (nt < nt_used) {
                    const uint4& Bv = (r < 2) ? B0[nt] : B1[nt];
                    const uint32_t b0 = (r & 1) ? Bv.z : Bv.x;
                    const uint32_t b1 = (r & 1) ? Bv.w : Bv.y;
                    mma_bf16_16816(d[nt], a, b0, b1);
                }
            }
        }
    }
}

struct RowChunk {
    uint4 qa, qb;
    uint32_t sa, sb;
};

__device__ __forceinline__ RowChunk load_rows(const uint8_t* ra, const uint8_t* rb, const uint8_t* sa,
                                              const uint8_t* sb, int ch, int c)
{
    RowChunk r;
    r.qa = ldg_stream_u4(ra + ch * 64 + c * 16);
    r.qb = ldg_stream_u4(rb + ch * 64 + c * 16);
    r.sa = ldg_u16(sa + ch * 8 + c * 2);
    r.sb = ldg_u16(sb + ch * 8 + c * 2);
    return r;
}

// ---------------------------------------------------------------- gate_up
//
// Work item = (active expert, 8 gate rows n0..n0+7 + the matching 8 up rows).
// A rows 0..7 are gate rows, rows 8..15 the up rows, so each thread ends with
// gate and up of the same (row, pair) in d[.][0/1] and d[.][2/3].  The NW warps
// of the CTA split K; partial sums are reduced in shared memory in warp order.
template <int NW>
__global__ void __launch_bounds__(NW * 32) decode_gate_up_kernel(
    const uint16_t* __restrict__ x_t16, const int32_t* __restrict__ sorted, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ active, const int32_t* __restrict__ active_count,
    const uint8_t* __restrict__ w13c, const uint8_t* __restrict__ w13s, int32_t H, int32_t I, int32_t k,
    uint16_t* __restrict__ h_t16, uint32_t* status)
{
    static_assert(NW >= kNT, "one warp per n-tile in the epilogue");
    __shared__ uint2 lut_tab[256];
    __shared__ float red[NW][kNT][32][4];
    init_lut_table(lut_tab);
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int n_act = *active_count;
    const int tiles_per_expert = I / 8;
    const int nch = H / kChunk;
    const int64_t rowb = H / 4, srowb = H / 32;
    uint32_t lut_min = 0xFFFFFFFFu;

    for (int item = blockIdx.x; item < n_act * tiles_per_expert; item += gridDim.x) {
        const int e = active[item / tiles_per_expert];
        const int n0 = (item % tiles_per_expert) * 8;
        const int q0 = offsets[e], cnt = offsets[e + 1] - q0;
        const int64_t rg = (int64_t)e * 2 * I + n0 + g, ru = rg + I;
        const uint8_t* ra = w13c + rg * rowb;
        const uint8_t* rb = w13c + ru * rowb;
        const uint8_t* sa = w13s + rg * srowb;
        const uint8_t* sb = w13s + ru * srowb;

        for (int pg = 0; pg < cnt; pg += kPairsPerPass) {
            const int nt_used = min(kNT, (cnt - pg + 7) / 8);
            const uint16_t* brow[kNT];
            bool bval[kNT];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                const int j = pg + nt * 8 + g;
                bval[nt] = j < cnt;
                brow[nt] = bval[nt] ? x_t16 + (int64_t)(sorted[q0 + j] / k) * H : x_t16;
            }
            float d[kNT][4];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;

            int ch = warp;
            RowChunk cur;
            if (ch < nch) cur = load_rows(ra, rb, sa, sb, ch, c);
            for (; ch < nch; ch += NW) {
                RowChunk nxt;
                if (ch + NW < nch) nxt = load_rows(ra, rb, sa, sb, ch + NW, c);
                const uint2 la0 = lut_tab[cur.sa & 0xFF], la1 = lut_tab[cur.sa >> 8];
                const uint2 lb0 = lut_tab[cur.sb & 0xFF], lb1 = lut_tab[cur.sb >> 8];
                lut_min = min(lut_min, min(min(la0.x, la1.x), min(lb0.x, lb1.x)));
                chunk_mma<kNT>(d, cur.qa, cur.qb, la0, la1, lb0, lb1, brow, bval, nt_used, ch * kChunk + c * 64);
                cur = nxt;
            }

#pragma unroll
            for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
                for (int v = 0; v < 4; ++v) red[warp][nt][lane][v] = d[nt][v];
            __syncthreads();
            if (warp < nt_used) {
                const int nt = warp;
                float gs[2] = {0.f, 0.f}, us[2] = {0.f, 0.f};
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    gs[0] += red[w][nt][lane][0];
                    gs[1] += red[w][nt][lane][1];
                    us[0] += red[w][nt][lane][2];
                    us[1] += red[w][nt][lane][3];
                }
                const int pos = t16_pos(n0 + g);
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int j = pg + nt * 8 + 2 * c + v;
                    if (j < cnt) {
                        const float hv = silu_f(gs[v]) * us[v];
                        __nv_bfloat16 hb = __float2bfloat16_rn(hv);
                        h_t16[(int64_t)(q0 + j) * I + pos] = *reinterpret_cast<uint16_t*>(&hb);
                    }
                }
            }
            __syncthreads();
        }
    }
    if (lut_min == 0) flag_status(status, MOE_W2_DEV_BAD_SCALE);
}

// ---------------------------------------------------------------- down + combine
//
// CTA = 16 output rows m0..m0+15 of y for every token.  Warp w takes the
// active experts a = w, w+NW, ... in ascending order; for each it computes
// W_down[e][rows] . h over its pairs and adds weight * result into its own
// per-token accumulator (shared memory, one column at a time so duplicate
// tokens never race).  Finally the warps' accumulators are summed in warp order
// and rounded to bf16 once: a fixed summation order, no atomics.
template <int NW>
__global__ void __launch_bounds__(NW * 32) decode_down_kernel(
    const uint16_t* __restrict__ h_t16, const int32_t* __restrict__ sorted, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ active, const int32_t* __restrict__ active_count, const float* __restrict__ weights,
    const uint8_t* __restrict__ w2c, const uint8_t* __restrict__ w2s, int32_t H, int32_t I, int32_t k, int32_t T,
    uint16_t* __restrict__ y, uint32_t* status)
{
    __shared__ uint2 lut_tab[256];
    extern __shared__ float acc[];   // [NW][16][T]
    init_lut_table(lut_tab);
    for (int i = threadIdx.x; i < NW * 16 * T; i += NW * 32) acc[i] = 0.f;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int m0 = blockIdx.x * 16;
    const int n_act = *active_count;
    const int nch = I / kChunk;
    const int64_t rowb = I / 4, srowb = I / 32;
    float* my_acc = acc + warp * 16 * T;
    uint32_t lut_min = 0xFFFFFFFFu;

    for (int a = warp; a < n_act; a += NW) {
        const int e = active[a];
        const int q0 = offsets[e], cnt = offsets[e + 1] - q0;
        const int64_t r0 = (int64_t)e * H + m0 + g;
        const uint8_t* ra = w2c + r0 * rowb;
        const uint8_t* rb = w2c + (r0 + 8) * rowb;
        const uint8_t* sa = w2s + r0 * srowb;
        const uint8_t* sb = w2s + (r0 + 8) * srowb;

        for (int pg = 0; pg < cnt; pg += kPairsPerPass) {
            const int nt_used = min(kNT, (cnt - pg + 7) / 8);
            const uint16_t* brow[kNT];
            bool bval[kNT];
            int tok[kNT][2];
            float wt[kNT][2];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                const int j = pg + nt * 8 + g;
                bval[nt] = j < cnt;
                brow[nt] = bval[nt] ? h_t16 + (int64_t)(q0 + j) * I : h_t16;
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    const int jj = pg + nt * 8 + 2 * c + v;
                    const int p = (jj < cnt) ? sorted[q0 + jj] : 0;
                    tok[nt][v] = p / k;
                    wt[nt][v] = (jj < cnt) ? weights[p] : 0.f;
                }
            }
            float d[kNT][4];
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;

            RowChunk cur = load_rows(ra, rb, sa, sb, 0, c);
            for (int ch = 0; ch < nch; ++ch) {
                RowChunk nxt;
                if (ch + 1 < nch) nxt = load_rows(ra, rb, sa, sb, ch + 1, c);
                const uint2 la0 = lut_tab[cur.sa & 0xFF], la1 = lut_tab[cur.sa >> 8];
                const uint2 lb0 = lut_tab[cur.sb & 0xFF], lb1 = lut_tab[cur.sb >> 8];
                lut_min = min(lut_min, min(min(la0.x, la1.x), min(lb0.x, lb1.x)));
                chunk_mma<kNT>(d, cur.qa, cur.qb, la0, la1, lb0, lb1, brow, bval, nt_used, ch * kChunk + c * 64);
                cur = nxt;
            }

            // weighted scatter into the per-token accumulator, one pair column at a time
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                if (nt >= nt_used) break;
#pragma unroll
                for (int col = 0; col < 8; ++col) {
                    if (c == (col >> 1) && pg + nt * 8 + col < cnt) {
                        const int v = col & 1;
                        float* dst = my_acc + tok[nt][v];
                        dst[g * T] += wt[nt][v] * d[nt][v];
                        dst[(g + 8) * T] += wt[nt][v] * d[nt][2 + v];
                    }
                    __syncwarp();
                }
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 16 * T; i += NW * 32) {
        const int t = i >> 4, row = i & 15;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += acc[(w * 16 + row) * T + t];
        __nv_bfloat16 yb = __float2bfloat16_rn(s);
        y[(int64_t)t * H + m0 + row] = *reinterpret_cast<uint16_t*>(&yb);
    }
    if (lut_min == 0) flag_status(status, MOE_W2_DEV_BAD_SCALE);
}

constexpr int kGateUpWarps = 4;
constexpr int kDownWarps = 8;

}  // namespace

cudaError_t launch_decode(const uint16_t* x_t16, const int32_t* ids, const float* weights, const moe_w2_planes& w,
                          int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status,
                          cudaStream_t s, const PhaseEvents& ev)
{
    (void)ids;
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    const int64_t max_items = std::min<int64_t>(P, E) * (I / 8);
    static int occ_gu = 0;
    if (occ_gu == 0) {
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ_gu, decode_gate_up_kernel<kGateUpWarps>,
                                                                      kGateUpWarps * 32, 0);
        if (e != cudaSuccess) return e;
        if (occ_gu < 1) occ_gu = 1;
    }
    const int grid_gu = (int)std::min<int64_t>(max_items, (int64_t)sm_count() * occ_gu);
    cudaError_t e = ev.record(1, s);
    if (e != cudaSuccess) return e;
    decode_gate_up_kernel<kGateUpWarps><<<grid_gu, kGateUpWarps * 32, 0, s>>>(
        x_t16, ws.sorted, ws.offsets, ws.active, ws.active_count, w.w13_codes, w.w13_scales, H, I, k, ws.h,
        status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = ev.record(2, s);
    if (e != cudaSuccess) return e;

    const size_t smem = sizeof(float) * kDownWarps * 16 * T;
    decode_down_kernel<kDownWarps><<<H / 16, kDownWarps * 32, smem, s>>>(
        ws.h, ws.sorted, ws.offsets, ws.active, ws.active_count, weights, w.w2_codes, w.w2_scales, H, I, k, T, y,
        status);
    return cudaGetLastError();
}

}  // namespace moe_w2
