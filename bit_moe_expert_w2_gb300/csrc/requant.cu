// Load-time re-quantizer: modelopt NVFP4 (e2m1 x e4m3 block-16 x fp32 scale_2)
// -> sign-symmetric 2-bit codes + UE8M0 block-32 scales, bit-exact.
//
// vLLM-Moet, page "The v0.24.0 port", section "Our hooks", modelopt.py bullet:
// dequantize to f64 exactly (all three factors representable), re-quantize to
// the {-4,-1,1,4} codebook, UE8M0 block-32 output scales absorb scale_2.  The
// scale is the least-squares one (page "vLLM-Moet wiki", section "2-bit expert
// planes": the symmetric codebook is chosen at the same L2 error).
//
// Exact integer formulation used here (no floating point decides anything):
//   |x_i| = N_i * 2^c with N_i = n1_i * Q_h * 2^(f_h - c) an integer, where
//   n1 = 2|e2m1| in {0,1,2,3,4,6,8,12}, Q_h = e4m3 integer mantissa * scale_2
//   integer mantissa, f_h the half-block's binary exponent.  For a candidate u,
//   SSE(u) - sum x^2 = 4^u (32 + 15 A) - 2^(u+1) 2^c (S + 3 S4), where A counts
//   the elements at magnitude 4 (|x| > 2.5 * 2^u) and S, S4 sum N over all /
//   over those elements.  Scaled by 4^-e (e = min(c, lo)) both terms are
//   integers below 2^112 and are compared in 128-bit arithmetic.
// Candidate window: u in [floor(log2 min|x|) - 5, floor(log2 max|x|) + 1] clamped
// to [-126, 125] holds the minimiser over all u (above it every code moves away
// from every element; below it all nonzero elements saturate and the error grows
// as u falls).  Ties go to the smaller u, an exact code tie to magnitude 1, and
// the code's sign is the element's sign bit.
//
// All elements of a half-block share Q_h and f_h, so an element's threshold
// depends only on its e2m1 magnitude class (7 nonzero classes per half): the
// kernel counts classes once (SWAR over nibbles), computes each class's
// threshold exponent tau (the largest u at which it is at magnitude 4) once, and
// evaluates each candidate from 14 integer comparisons against tau.
//
// MXFP4 (page "The v0.24.0 port", section "Our hooks", mxfp4.py bullet; page
// "vLLM-Moet wiki": FP4 experts load by a codes remap): e2m1 elements with one
// UE8M0 byte s per 32, x_i = e2m1_i * 2^(s-127), byte 255 = NaN.  This is the
// NVFP4 case with Q_h = 1 and f_h = s - 128 in both halves, so the same kernel
// serves it; the codes come out as a function of the e2m1 codes alone and the
// byte moves with s, which is the remap.
//
// Zero-sign balancing (page "vLLM-Moet wiki", the Kimi-K2.7 paragraph: an export
// writing every exact zero as +0 biases the codes): with the option, the exact
// zeros of a block take the signs +,-,+,- ... in element order.  A zero is at
// magnitude 1 for every u, so the scale search is unchanged.
#include <algorithm>

#include "common.cuh"

namespace moe_w2 {

namespace {

__device__ __forceinline__ int n1_of_class(int v)
{
    // 2 * |e2m1| for magnitude bits v = 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6
    return (v < 4) ? v : (v == 4 ? 4 : (v == 5 ? 6 : (v == 6 ? 8 : 12)));
}

// Number of nibbles of w (low 3 bits) equal to v, for v in 1..7.
__device__ __forceinline__ int count_class(uint32_t w, uint32_t v)
{
    const uint32_t t = (w & 0x77777777u) ^ (v * 0x11111111u);
    const uint32_t z = ~(t + 0x77777777u) & 0x88888888u;
    return __popc(z);
}

// 8 nibbles -> 8 two-bit codes (16 bits).  ge: bit 3 of each nibble = magnitude 4;
// sg: bit 3 of each nibble = negative.
__device__ __forceinline__ uint32_t pack_codes(uint32_t ge, uint32_t sg)
{
    uint32_t x = ((ge >> 3) & 0x11111111u) | ((sg >> 2) & 0x22222222u);
    x = (x | (x >> 2)) & 0x0F0F0F0Fu;
    x = (x | (x >> 4)) & 0x00FF00FFu;
    x = (x | (x >> 8)) & 0x0000FFFFu;
    return x;
}

__device__ __forceinline__ int floor_log2_u64(uint64_t v) { return 63 - __clzll((long long)v); }

struct Half {
    uint32_t Q;      // e4m3 integer mantissa * scale_2 integer mantissa (0 if the scale is 0)
    int f;           // binary exponent of the unit of Q (|x| = n1 * Q * 2^f)
    uint32_t neg;    // e4m3 sign
    bool nan;
};

__device__ __forceinline__ Half decode_half(uint32_t b, uint32_t S, int es)
{
    Half h;
    const uint32_t E4 = (b >> 3) & 15u, m = b & 7u;
    h.nan = (E4 == 15u && m == 7u);
    h.neg = (b >> 7) & 1u;
    const uint32_t M = E4 ? (8u + m) : m;
    const int e4 = E4 ? (int)E4 - 10 : -9;   // value = M * 2^e4
    h.Q = M * S;
    h.f = e4 + es - 1;                       // n1 = 2|e2m1| carries the extra factor 2
    return h;
}

// Zero-sign balancing of one block: w = the 4 words of 8 nibbles (element
// order), zq = per half whether its scale is 0 (every element exactly zero);
// sg = sign bits (bit 3 of each nibble), returned with the zeros' signs set to
// +,-,+,- ... in element order.
__device__ __forceinline__ void balance_zero_signs(const uint32_t (&w)[4], const bool (&zq)[2], uint32_t (&sg)[4])
{
    uint32_t par = 0;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t z = zq[wi >> 1] ? 0x88888888u : (~((w[wi] & 0x77777777u) + 0x77777777u) & 0x88888888u);
        uint32_t bal = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t bit = 1u << (4 * k + 3);
            if (z & bit) {
                bal |= par ? bit : 0u;
                par ^= 1u;
            }
        }
        sg[wi] = (sg[wi] & ~z) | bal;
    }
}

// kMx = false: NVFP4 (scale bytes = two e4m3 per block, scale_2 per tensor);
// kMx = true: MXFP4 (scale bytes = one UE8M0 per block, scale_2 unused).
template <bool kMx>
__global__ void __launch_bounds__(256) requant_kernel(const uint8_t* __restrict__ e2m1,
                                                      const uint8_t* __restrict__ scale_bytes,
                                                      const float* __restrict__ scale_2, int64_t n_blocks,
                                                      int64_t blocks_per_tensor, uint32_t balance,
                                                      uint8_t* __restrict__ codes, uint8_t* __restrict__ ue8m0,
                                                      uint32_t* status)
{
    uint32_t bad_any = 0;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < n_blocks;
         blk += (int64_t)gridDim.x * blockDim.x) {
        const uint4 nib = ldg_stream_u4(e2m1 + blk * 16);
        Half hf[2];
        bool s2_bad = false;
        if constexpr (kMx) {
            const uint32_t sb = __ldg(scale_bytes + blk);
            hf[0].Q = 1u;
            hf[0].f = (int)sb - 128;   // n1 = 2|e2m1| carries the extra factor 2
            hf[0].neg = 0u;
            hf[0].nan = sb == 0xFFu;
            hf[1] = hf[0];
        } else {
            const int64_t tensor = blk / blocks_per_tensor;
            const uint32_t sbits = __float_as_uint(__ldg(scale_2 + tensor));
            const uint32_t sc = ldg_u16(scale_bytes + blk * 2);
            // scale_2 = S * 2^es
            const uint32_t sE = (sbits >> 23) & 0xFFu, sM = sbits & 0x7FFFFFu;
            s2_bad = (sbits >> 31) != 0u || sE == 0xFFu || (sE == 0u && sM == 0u);
            const uint32_t S = sE ? (sM | 0x800000u) : sM;
            const int es = sE ? (int)sE - 150 : -149;
            hf[0] = decode_half(sc & 0xFFu, S, es);
            hf[1] = decode_half(sc >> 8, S, es);
        }
        if (s2_bad || hf[0].nan || hf[1].nan) {
            *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(0u, 0u);
            ue8m0[blk] = 0;
            bad_any = 1;
            continue;
        }

        const uint32_t w[4] = {nib.x, nib.y, nib.z, nib.w};   // half 0 = w[0..1], half 1 = w[2..3]

        // class counts per half, and the unit exponent c
        int cntv[2][8];
        bool any[2];
        for (int h = 0; h < 2; ++h) {
            int tot = 0;
#pragma unroll
            for (int v = 1; v < 8; ++v) {
                cntv[h][v] = count_class(w[2 * h], v) + count_class(w[2 * h + 1], v);
                tot += cntv[h][v];
            }
            any[h] = tot > 0 && hf[h].Q != 0u;
        }

        int u;
        int v0[2] = {8, 8};   // smallest magnitude class at magnitude 4, per half
        if (!any[0] && !any[1]) {
            u = -126;
        } else {
            const int c = (any[0] && any[1]) ? min(hf[0].f, hf[1].f) : (any[0] ? hf[0].f : hf[1].f);
            uint64_t Qs[2];
            uint64_t nmax = 0, nmin = ~0ull;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                Qs[h] = any[h] ? ((uint64_t)hf[h].Q << (hf[h].f - c)) : 0ull;
                if (!any[h]) continue;
                int vmax = 0, vmin = 8;
#pragma unroll
                for (int v = 7; v >= 1; --v)
                    if (cntv[h][v] && vmax == 0) vmax = v;
#pragma unroll
                for (int v = 1; v < 8; ++v)
                    if (cntv[h][v] && vmin == 8) vmin = v;
                nmax = max(nmax, (uint64_t)n1_of_class(vmax) * Qs[h]);
                nmin = min(nmin, (uint64_t)n1_of_class(vmin) * Qs[h]);
            }
            const int m = floor_log2_u64(nmax) + c, mlo = floor_log2_u64(nmin) + c;
            // Threshold of each class: the largest u at which it is at magnitude 4.
            // |x| > 2.5 * 2^u  <=>  N > 5 * 2^(u-c-1); with L = floor(log2 N) the largest
            // k with 5 * 2^k < N is L-2 when 4N > 5 * 2^L, else L-3; tau = k + c + 1.
            int tau[2][8];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int v = 1; v < 8; ++v) {
                    const uint64_t N = (uint64_t)n1_of_class(v) * Qs[h];
                    if (!any[h] || N == 0) {
                        tau[h][v] = -100000;
                        continue;
                    }
                    const int L = floor_log2_u64(N);
                    tau[h][v] = ((N << 2) > (5ull << L) ? L - 2 : L - 3) + c + 1;
                }
            int hi = min(125, max(-126, m + 1));
            int lo = min(hi, max(-126, mlo - 5));
            {
                // Dominated low candidates.  While u <= tau_min every nonzero element
                // is at magnitude 4, so SSE(u) = f(2^u) with f(e) = sum (a_i - 4e)^2 +
                // n0 e^2, minimal at e* = 4 sum a / (16 n + n0); f(2e) < f(e) exactly
                // when e < 2 e* / 3, and SSE(u+1) <= f(2^(u+1)) (nearest codes never do
                // worse than magnitude 4).  Hence every u <= tau_min with
                // 3 (16 n + n0) 2^u < 8 sum a is strictly worse than u+1 and the search
                // can start at min(tau_min + 1, smallest u without that property).
                int n_nz = 0, tau_min = 1 << 20, tau_max = -(1 << 20);
                uint64_t S_nz = 0;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int v = 1; v < 8; ++v)
                        if (any[h] && cntv[h][v]) {
                            n_nz += cntv[h][v];
                            S_nz += (uint64_t)cntv[h][v] * ((uint64_t)n1_of_class(v) * Qs[h]);
                            tau_min = min(tau_min, tau[h][v]);
                            tau_max = max(tau_max, tau[h][v]);
                        }
                // smallest e with D 2^e >= Num (|x| = N 2^c, so sum a = S_nz 2^c, u = e + c)
                const uint64_t D = 3ull * (uint64_t)(16 * n_nz + (32 - n_nz));
                const uint64_t Num = 8ull * S_nz;
                int e = floor_log2_u64(Num) - floor_log2_u64(D) - 1;
                auto reaches = [&](int ee) {
                    return ee >= 0 ? ((unsigned __int128)D << ee) >= (unsigned __int128)Num
                                   : (unsigned __int128)D >= ((unsigned __int128)Num << (-ee));
                };
                while (!reaches(e)) ++e;
                const int lo_new = min(tau_min + 1, e + c);
                lo = min(hi, max(lo, lo_new));
                // Dominated high candidates.  Above tau_max every element is at
                // magnitude 1, SSE(u) = g(2^u) with g(e) = sum over all 32 of (a_i - e)^2;
                // g(e/2) < g(e) exactly when 24 e > sum a, and SSE(u-1) <= g(2^(u-1)).
                // Hence every u > tau_max with 24 2^u > sum a is strictly worse than u-1:
                // the search can stop at max(tau_max, largest u with 24 2^u <= sum a).
                int f = floor_log2_u64(S_nz) - 4;   // largest f with 24 2^f <= S_nz (f >= L-5)
                auto fits = [&](int ff) {
                    return ff >= 0 ? ((unsigned __int128)24 << ff) <= (unsigned __int128)S_nz
                                   : (unsigned __int128)24 <= ((unsigned __int128)S_nz << (-ff));
                };
                while (!fits(f)) --f;
                while (fits(f + 1)) ++f;
                hi = max(lo, min(hi, max(tau_max, f + c)));
            }
            if (lo == hi) {
                u = lo;
            } else {
                const int eref = min(c, lo);
                const int C1 = c - eref + 1;
                uint64_t S_all = 0;
                uint64_t cN[2][8];   // count * N of each class
                int cc[2][8];        // count of each class
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int v = 1; v < 8; ++v) {
                        cc[h][v] = any[h] ? cntv[h][v] : 0;
                        cN[h][v] = (uint64_t)cc[h][v] * ((uint64_t)n1_of_class(v) * Qs[h]);
                        S_all += cN[h][v];
                    }
                __int128 best = 0;
                int best_u = lo;
                for (int cand = lo; cand <= hi; ++cand) {
                    const int U = cand - eref;
                    int A = 0;
                    uint64_t S4 = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int v = 1; v < 8; ++v)
                            if (tau[h][v] >= cand) {
                                A += cc[h][v];
                                S4 += cN[h][v];
                            }
                    const __int128 t1 = (__int128)(32 + 15 * A) << (2 * U);
                    const __int128 t2 = (__int128)(S_all + 3 * S4) << (U + C1);
                    const __int128 G = t1 - t2;
                    if (cand == lo || G < best) {
                        best = G;
                        best_u = cand;
                    }
                }
                u = best_u;
            }
            // magnitude-4 classes at the chosen u: the smallest class whose threshold reaches u
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (!any[h]) continue;
                int vv = 8;
#pragma unroll
                for (int v = 7; v >= 1; --v)
                    if (tau[h][v] >= u) vv = v;
                v0[h] = vv;
            }
        }

        // codes: magnitude 4 iff class >= v0, sign = e2m1 sign xor e4m3 sign
        uint32_t sg[4];
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) sg[wi] = (w[wi] ^ (hf[wi >> 1].neg ? 0x88888888u : 0u)) & 0x88888888u;
        if (balance) {
            const bool zq[2] = {hf[0].Q == 0u, hf[1].Q == 0u};
            balance_zero_signs(w, zq, sg);
        }
        uint32_t out[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t half16[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int wi = 2 * q + j, h = q;
                const uint32_t ww = w[wi];
                const uint32_t ge = ((ww & 0x77777777u) + (uint32_t)(8 - v0[h]) * 0x11111111u) & 0x88888888u;
                half16[j] = pack_codes(ge, sg[wi]);
            }
            out[q] = half16[0] | (half16[1] << 16);
        }
        *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(out[0], out[1]);
        ue8m0[blk] = (uint8_t)(u + 127);
    }
    if (bad_any) flag_status(status, MOE_W2_DEV_BAD_NVFP4);
}

}  // namespace

// ------------------------------------------------------------------ FP8 block-128
//
// vLLM-Moet, page "The v0.24.0 port", section "Our hooks", fp8.py bullet: the FP8
// block-quant loader re-quantizes fp8 weights with f32 block-128 scales to the
// same codebook in float64.  Element x_i = e4m3_i * S, S the f32 scale of the
// 128 x 128 block holding it; all 32 elements of an output block share S.
//
// Exact integer form: e4m3 magnitude = A_i * 2^-9 with A_i an integer below 2^18
// (subnormals m, normals (8 + m) 2^(e-1)); S = s_m * 2^s_e with s_m the f32
// integer significand.  So |x_i| = N_i * 2^c, N_i = A_i s_m < 2^42, c = s_e - 9.
// For candidate u an element is at magnitude 4 iff N_i 2^(c - u + 1) > 5, and
//   SSE(u) - sum x^2 = 4^u V(u) - 2^(u + 1 + c) W(u),
// V = sum of v_i^2 (1 or 16), W = sum of N_i v_i (v_i 1 or 4).  Both terms are
// scaled by 2^-e0, e0 = min(2 lo, lo + 1 + c), to integers below 2^104 and
// compared in 128-bit arithmetic, candidates ascending, strictly smaller wins.
// The window [floor(log2 min|x|) - 5, floor(log2 max|x|) + 1] clamped to
// [-126, 125] is the one the NVFP4 path uses (same argument); within it every
// shift below stays in range (c - u + 1 <= 6, u - c - 1 <= 43).
__global__ void __launch_bounds__(256) requant_fp8_kernel(const uint8_t* __restrict__ w8,
                                                          const float* __restrict__ scales, int64_t n_blocks,
                                                          int64_t rows, int64_t bpr, int64_t srows, int64_t scols,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ ue8m0,
                                                          uint32_t* status)
{
    uint32_t bad = 0;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n_blocks;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = g / (rows * bpr), r = (g / bpr) % rows, b = g % bpr;
        const uint32_t sb = __float_as_uint(__ldg(scales + (t * srows + r / 128) * scols + (b * 32) / 128));
        const uint4 q0 = __ldg(reinterpret_cast<const uint4*>(w8 + g * 32));
        const uint4 q1 = __ldg(reinterpret_cast<const uint4*>(w8 + g * 32 + 16));
        const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        // NaN codes (S.1111.111) anywhere, or a scale that is not positive finite
        uint32_t nan = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t t7 = (wv[k] & 0x7F7F7F7Fu) + 0x01010101u;   // 0x80 per byte exactly when its low 7 bits are all ones
            nan |= t7 & 0x80808080u;
        }
        if (nan != 0 || sb == 0u || sb >= 0x7F800000u) {
            *reinterpret_cast<uint2*>(codes + g * 8) = make_uint2(0u, 0u);
            ue8m0[g] = 0;
            bad = 1;
            continue;
        }
        const uint32_t es = sb >> 23;
        const uint64_t sm = es == 0u ? (uint64_t)(sb & 0x7FFFFFu) : (uint64_t)((sb & 0x7FFFFFu) | 0x800000u);
        const int c = (es == 0u ? -149 : (int)es - 150) - 9;
        uint64_t N[32];
        uint32_t negm = 0;
        uint64_t nmax = 0, nmin = ~0ull;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t byte = (wv[i >> 2] >> (8 * (i & 3))) & 0xFFu;
            const uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
            const uint64_t A = e == 0u ? (uint64_t)m : (uint64_t)(8u + m) << (e - 1u);
            N[i] = A * sm;
            negm |= (byte >> 7) << i;
            nmax = max(nmax, N[i]);
            if (N[i] != 0ull) nmin = min(nmin, N[i]);
        }
        int best_u;
        if (nmax == 0ull) {
            best_u = -126;   // every candidate costs 32 * 4^u: the smallest scale
        } else {
            const int mhi = 63 - __clzll((long long)nmax) + c, mlo = 63 - __clzll((long long)nmin) + c;
            const int hi = min(125, max(-126, mhi + 1));
            const int lo = min(hi, max(-126, mlo - 5));
            const int e0 = min(2 * lo, lo + 1 + c);
            __int128 best = 0;
            best_u = lo;
            for (int u = lo; u <= hi; ++u) {
                const int d = c - u + 1;
                uint32_t V = 0;
                unsigned __int128 W = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const bool four = d >= 0 ? (N[i] << d) > 5ull : N[i] > (5ull << (-d));
                    V += four ? 16u : 1u;
                    W += four ? (unsigned __int128)N[i] * 4u : (unsigned __int128)N[i];
                }
                const __int128 G = ((__int128)V << (2 * u - e0)) - (__int128)(W << (u + 1 + c - e0));
                if (u == lo || G < best) {
                    best = G;
                    best_u = u;
                }
            }
        }
        // codes at the chosen scale: 2-bit c = sign << 1 | magnitude 4
        const int d = c - best_u + 1;
        uint32_t lo_w = 0, hi_w = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const bool four = nmax != 0ull && (d >= 0 ? (N[i] << d) > 5ull : N[i] > (5ull << (-d)));
            const uint32_t code = (((negm >> i) & 1u) << 1) | (four ? 1u : 0u);
            if (i < 16) lo_w |= code << (2 * i);
            else hi_w |= code << (2 * (i - 16));
        }
        *reinterpret_cast<uint2*>(codes + g * 8) = make_uint2(lo_w, hi_w);
        ue8m0[g] = (uint8_t)(best_u + 127);
    }
    if (bad) flag_status(status, MOE_W2_DEV_BAD_NVFP4);
}

cudaError_t launch_requant(const uint8_t* e2m1, const uint8_t* e4m3, const float* scale_2, int64_t n, int64_t rows,
                           int64_t K, uint32_t options, uint8_t* codes, uint8_t* ue8m0, uint32_t* status,
                           cudaStream_t s)
{
    const int64_t bpt = rows * (K / 32);
    const int64_t nb = n * bpt;
    if (nb == 0) return cudaSuccess;
    const int64_t want = (nb + 255) / 256;
    const int grid = (int)std::min<int64_t>(want, (int64_t)sm_count() * 8);
    requant_kernel<false><<<grid, 256, 0, s>>>(e2m1, e4m3, scale_2, nb, bpt, options & MOE_W2_REQUANT_BALANCE_ZERO_SIGNS,
                                               codes, ue8m0, status);
    return cudaGetLastError();
}

cudaError_t launch_requant_mxfp4(const uint8_t* e2m1, const uint8_t* scales, int64_t n, int64_t rows, int64_t K,
                                 uint32_t options, uint8_t* codes, uint8_t* ue8m0, uint32_t* status, cudaStream_t s)
{
    const int64_t nb = n * rows * (K / 32);
    if (nb == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>((nb + 255) / 256, (int64_t)sm_count() * 8);
    requant_kernel<true><<<grid, 256, 0, s>>>(e2m1, scales, nullptr, nb, nb, options & MOE_W2_REQUANT_BALANCE_ZERO_SIGNS,
                                              codes, ue8m0, status);
    return cudaGetLastError();
}

cudaError_t launch_requant_fp8(const uint8_t* w8, const float* scales, int64_t n, int64_t rows, int64_t K,
                               uint8_t* codes, uint8_t* ue8m0, uint32_t* status, cudaStream_t s)
{
    const int64_t bpr = K / 32, n_blocks = n * rows * bpr;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n_blocks + 255) / 256, (int64_t)sm_count() * 16));
    requant_fp8_kernel<<<grid, 256, 0, s>>>(w8, scales, n_blocks, rows, bpr, (rows + 127) / 128, (K + 127) / 128, codes,
                                            ue8m0, status);
    return cudaGetLastError();
}

}  // namespace moe_w2
