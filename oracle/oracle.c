/*
 * CPU oracle for the 2-bit sign-symmetric MoE layer (vLLM-Moet) and its NVFP4
 * re-quantizer.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never does.
 *
 * Plain loops in f64 (and exact 128-bit integer sums where an L2 comparison has
 * to be exact).  No blocking, no fusion, no reordering beyond what each
 * definition states.  Shares no source with the CUDA library.
 *
 * The same source builds twice: single-threaded, and with OpenMP, where the
 * loops over independent blocks (requant) and tokens (forward) run on several
 * threads.  Every block and every token is computed by one thread with the
 * same sequence of operations, so both builds give bitwise identical results.
 *
 * Sources (vLLM-Moet pages):
 *   [wiki]  "vLLM-Moet wiki", section "2-bit expert planes": codebook {-4,-1,1,4},
 *           sign-symmetric, chosen at the same L2 error.
 *   [port]  "The v0.24.0 port", section "Our hooks", modelopt.py bullet: NVFP4 =
 *           e2m1 codes x e4m3 block-16 scales x per-tensor scale_2, dequantized
 *           to f64 exactly (all three factors representable), re-quantized to
 *           the sign-symmetric codebook with UE8M0 block-32 output scales that
 *           absorb scale_2.
 *   [port]  same section, BASE-cache bullet: codes + UE8M0 scales, four
 *           sections per expert slot.
 *   [port]  same section, "Deterministic unpermute" bullet: valid sorted ids are
 *           a permutation of token*top_k+j; outputs are placed per pair and
 *           summed over j in a fixed order.
 *
 * Readings taken where the pages are silent:
 *   R1 code order: 2-bit code c = (sign << 1) | magnitude, i.e. 0:+1 1:+4 2:-1 3:-4.
 *   R2 packing: 4 codes per byte along K, element 4b+q in bits 2q..2q+1 of byte b.
 *   R3 scale search: the UE8M0 exponent u in [-126,125] that minimises the exact
 *      L2 error with every element at its nearest code; ties go to the smaller u.
 *   R4 nearest code: magnitude 4 iff |x| > 2.5*2^u (a tie goes to magnitude 1);
 *      the code's sign is the sign bit of x, so -0 maps to -1.
 *   R5 invalid input: scale_2 not a positive finite number, or an e4m3 NaN in
 *      the block -> codes 0x00 and scale byte 0 for the block, status bit 4.
 *   R6 forward: gate rows 0..I-1 and up rows I..2I-1 of w13; h = bf16(SiLU(g)*u);
 *      the router weight multiplies the down projection; y = bf16(sum over j in
 *      j order); all sums in f64.  Expert ids outside [0,E) contribute nothing
 *      (status bit 1); a UE8M0 byte outside [1,252] zeroes its block (bit 2).
 *   R9 expert cache ("vLLM-Moet wiki", BASE-cache paragraph; "The v0.24.0 port",
 *      "Our hooks", BASE-cache bullet): the planes hold S slots and a table maps
 *      each routed id in [0, n_route) to its slot, negative when the expert is
 *      not resident.  A missing expert's pair contributes nothing and is counted
 *      (no status bit); an id outside [0, n_route) or a slot >= S is an invalid
 *      id (bit 1).
 *   R10 MXFP4 checkpoints ("vLLM-Moet wiki": FP4 experts load by a codes remap;
 *      "The v0.24.0 port", "Our hooks", mxfp4.py bullet): e2m1 elements with
 *      one UE8M0 scale byte per 32, x_i = e2m1_i * 2^(s-127), byte 255 = NaN
 *      (invalid block, bit 4).  The planes follow the same rule as R3/R4; as
 *      the scale is a power of two the codes depend on the e2m1 codes alone and
 *      the output byte is the input byte shifted, hence "remap".
 *   R11 zero-sign balancing (page "vLLM-Moet wiki", the Kimi-K2.7 paragraph: an
 *      export that writes every exact zero as +0 biases the codes): with the
 *      option on, the exact zeros of a block take the signs +,-,+,- ... in
 *      element order instead of their sign bits; nothing else changes (a zero
 *      is at magnitude 1 for every u, so the scale search does not see it).
 *   R12 the FP4 layer (page "vLLM-Moet wiki", "The kernels" and "FP4 recovery":
 *      moe_w4_mm, the same forward over the NVFP4 experts): every weight is
 *      e2m1 x e4m3 (its 16-element block) x scale_2 (per tensor: gate, up and
 *      down of each expert have their own), dequantised exactly in f64; the
 *      rest is R6.  An e4m3 NaN scale zeroes its 16 elements (bit 2).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
/* independent iterations on all threads, status bits OR-reduced: blocks of 32
 * elements are handed out 256 at a time, tokens one at a time */
#define ORACLE_PARALLEL_FOR_BLOCKS _Pragma("omp parallel for schedule(dynamic, 256) reduction(|:st)")
#define ORACLE_PARALLEL_FOR_TOKENS _Pragma("omp parallel for schedule(dynamic, 1) reduction(|:st)")
#else
#define ORACLE_PARALLEL_FOR_BLOCKS
#define ORACLE_PARALLEL_FOR_TOKENS
#endif

#define ORACLE_BAD_EXPERT_ID 1u
#define ORACLE_BAD_SCALE 2u
#define ORACLE_BAD_NVFP4 4u

typedef unsigned __int128 u128;

int oracle_version(void) { return 1; }

/* Threads the parallel loops use (1 in the single-threaded build). */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void oracle_fail(const char *what)
{
    fprintf(stderr, "oracle: internal check failed: %s\n", what);
    abort();
}

/* ---------------------------------------------------------------- value tables */

/* e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. */
double oracle_e2m1_value(unsigned nib)
{
    unsigned s = (nib >> 3) & 1u, e = (nib >> 1) & 3u, m = nib & 1u;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - 1);
    return s ? -mag : mag;
}

/* e4m3fn: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa;
 * S.1111.111 is NaN, there is no infinity. */
double oracle_e4m3_value(unsigned b)
{
    unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* The sign-symmetric codebook under reading R1. */
double oracle_code_value(unsigned c)
{
    static const double v[4] = {1.0, 4.0, -1.0, -4.0};
    return v[c & 3u];
}

/* UE8M0 byte s -> 2^(s-127); the forward accepts s in [1,252] only. */
static int ue8m0_valid(unsigned s) { return s >= 1 && s <= 252; }

double oracle_bf16_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* f64 -> bf16, one rounding, to nearest with ties to even. */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int ex;
    (void)frexp(a, &ex);                 /* a in [2^(ex-1), 2^ex) */
    int q = (ex - 1 >= -126) ? ex - 8 : -133;   /* quantum: 8 significant bits, or subnormal */
    double r = nearbyint(ldexp(a, -q)) ;  /* default rounding mode: to nearest even */
    double rv = ldexp(r, q);
    float f = (float)rv;                 /* exact (<= 8 significant bits) or overflow to inf */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    if (isinf(f)) return sign | 0x7F80;
    return sign | (uint16_t)(bits >> 16);
}

/* ------------------------------------------------------------------ requant */

/* Re-quantisation of one block of 32 exact values (each an f64 with at most 53
 * significant bits, here at most 30) -> 8 code bytes and one UE8M0 byte, by
 * readings R3 and R4.  Shared by the NVFP4 and FP8 loaders, which differ only
 * in how they dequantise. */
static void search_block(const double *x, int balance_zeros, uint8_t *codes_out, uint8_t *scale_out)
{
    double a[32];
    int neg[32];
    double amax = 0.0, min_nz = INFINITY;
    int zeros = 0;
    for (int i = 0; i < 32; ++i) {
        neg[i] = signbit(x[i]) ? 1 : 0;
        a[i] = fabs(x[i]);
        if (balance_zeros && a[i] == 0.0) neg[i] = (zeros++) & 1;   /* reading R11 */
        if (a[i] > amax) amax = a[i];
        if (a[i] > 0.0 && a[i] < min_nz) min_nz = a[i];
    }

    int u;
    if (amax == 0.0) {
        u = -126;   /* every candidate costs 32*4^u: the smallest scale wins */
    } else {
        /* Candidate window.  u > m+1 only moves every code further from every x;
         * below 2^u < min_nz/12 the error grows as u falls (all nonzero
         * elements saturate at 4*2^u).  lo = floor(log2 min_nz) - 5 is below
         * that point, so [lo, m+1] holds the minimiser over all u in [-126,125]. */
        int ex;
        (void)frexp(amax, &ex);
        int m = ex - 1;
        (void)frexp(min_nz, &ex);
        int mlo = ex - 1;
        int hi = m + 1, lo = mlo - 5;
        if (hi > 125) hi = 125;
        if (hi < -126) hi = -126;
        if (lo < -126) lo = -126;
        if (lo > hi) lo = hi;

        if (lo == hi) {
            u = lo;
        } else {
            /* |x_i| = N_i * 2^c with N_i integer; c = lowest set bit of the block. */
            int c = 1 << 30;
            for (int i = 0; i < 32; ++i) {
                if (a[i] == 0.0) continue;
                int e2;
                double f = frexp(a[i], &e2);
                uint64_t M = (uint64_t)ldexp(f, 53);
                int tz = __builtin_ctzll(M);
                int low = e2 - 53 + tz;
                if (low < c) c = low;
            }
            int e0 = (c < lo) ? c : lo;   /* common unit 2^e0 for every candidate */
            if (c - e0 > 8) oracle_fail("requant: unit shift");
            uint64_t A[32];
            for (int i = 0; i < 32; ++i) {
                double n = ldexp(a[i], -c);
                if (n >= 9007199254740992.0) oracle_fail("requant: mantissa range");
                A[i] = ((uint64_t)n) << (c - e0);
            }
            u128 best = 0;
            int best_u = lo;
            for (int cand = lo; cand <= hi; ++cand) {
                if (cand - e0 > 58) oracle_fail("requant: candidate range");
                double thr = 2.5 * ldexp(1.0, cand);
                u128 sse = 0;
                for (int i = 0; i < 32; ++i) {
                    uint64_t mag = (a[i] > thr) ? 4u : 1u;
                    uint64_t V = mag << (cand - e0);
                    uint64_t d = (A[i] > V) ? A[i] - V : V - A[i];
                    sse += (u128)d * (u128)d;
                }
                if (cand == lo || sse < best) {
                    best = sse;
                    best_u = cand;
                }
            }
            u = best_u;
        }
    }

    double thr = 2.5 * ldexp(1.0, u);
    memset(codes_out, 0, 8);
    for (int i = 0; i < 32; ++i) {
        unsigned mag4 = (a[i] > thr) ? 1u : 0u;
        unsigned code = ((unsigned)neg[i] << 1) | mag4;
        codes_out[i / 4] |= (uint8_t)(code << (2 * (i % 4)));
    }
    *scale_out = (uint8_t)(u + 127);
}

/* One block of 32 NVFP4 elements -> 8 code bytes and one UE8M0 byte. */
static uint32_t requant_block(const uint8_t *nib_bytes, const uint8_t *e4m3_pair, float scale_2, int balance,
                              uint8_t *codes_out, uint8_t *scale_out)
{
    double s2 = (double)scale_2;
    double sc[2] = {oracle_e4m3_value(e4m3_pair[0]), oracle_e4m3_value(e4m3_pair[1])};
    if (!(s2 > 0.0) || isinf(s2) || isnan(sc[0]) || isnan(sc[1])) {
        memset(codes_out, 0, 8);
        *scale_out = 0;
        return ORACLE_BAD_NVFP4;
    }
    /* Exact f64 dequantisation: each product has at most 2+4+24 significant bits. */
    double x[32];
    for (int i = 0; i < 32; ++i) {
        unsigned nib = (nib_bytes[i / 2] >> (4 * (i % 2))) & 0xFu;
        x[i] = oracle_e2m1_value(nib) * sc[i / 16] * s2;
    }
    search_block(x, balance, codes_out, scale_out);
    return 0;
}

/* One block of 32 MXFP4 elements (reading R10) -> 8 code bytes and one UE8M0 byte. */
static uint32_t requant_block_mx(const uint8_t *nib_bytes, uint8_t s, int balance, uint8_t *codes_out,
                                 uint8_t *scale_out)
{
    if (s == 0xFFu) {
        memset(codes_out, 0, 8);
        *scale_out = 0;
        return ORACLE_BAD_NVFP4;
    }
    double x[32];
    for (int i = 0; i < 32; ++i) {
        unsigned nib = (nib_bytes[i / 2] >> (4 * (i % 2))) & 0xFu;
        x[i] = ldexp(oracle_e2m1_value(nib), (int)s - 127);   /* exact */
    }
    search_block(x, balance, codes_out, scale_out);
    return 0;
}

/* One block of 32 FP8 elements (e4m3fn bytes) under one f32 block scale -> 8
 * code bytes and one UE8M0 byte.  An e4m3 NaN in the block, or a scale that is
 * not a positive finite number, makes the block invalid (codes 0x00, scale
 * byte 0, status bit 4), as for NVFP4. */
static uint32_t requant_block_fp8(const uint8_t *e4m3_bytes, float scale, uint8_t *codes_out, uint8_t *scale_out)
{
    double s = (double)scale;
    int bad = !(s > 0.0) || isinf(s);
    double x[32];
    for (int i = 0; i < 32 && !bad; ++i) {
        double v = oracle_e4m3_value(e4m3_bytes[i]);
        if (isnan(v)) bad = 1;
        /* exact: at most 4 + 24 significant bits */
        x[i] = v * s;
    }
    if (bad) {
        memset(codes_out, 0, 8);
        *scale_out = 0;
        return ORACLE_BAD_NVFP4;
    }
    search_block(x, 0, codes_out, scale_out);
    return 0;
}

/* Option bit of the FP4 loaders: reading R11. */
#define ORACLE_BALANCE_ZERO_SIGNS 1u

/* Whole tensors: e2m1 [n][rows][K/2], e4m3 [n][rows][K/16], scale_2 [n]
 * -> codes [n][rows][K/4], ue8m0 [n][rows][K/32].  Returns status bits. */
uint32_t oracle_requant_ex(const uint8_t *e2m1, const uint8_t *e4m3, const float *scale_2,
                           int64_t n, int64_t rows, int64_t K, uint32_t options, uint8_t *codes, uint8_t *ue8m0)
{
    if (K % 32 != 0) return 0x80000000u;
    uint32_t st = 0;
    int64_t blocks_per_tensor = rows * (K / 32);
    int balance = (options & ORACLE_BALANCE_ZERO_SIGNS) != 0;
    ORACLE_PARALLEL_FOR_BLOCKS
    for (int64_t g = 0; g < n * blocks_per_tensor; ++g)
        st |= requant_block(e2m1 + g * 16, e4m3 + g * 2, scale_2[g / blocks_per_tensor], balance, codes + g * 8,
                            ue8m0 + g);
    return st;
}

uint32_t oracle_requant(const uint8_t *e2m1, const uint8_t *e4m3, const float *scale_2,
                        int64_t n, int64_t rows, int64_t K, uint8_t *codes, uint8_t *ue8m0)
{
    return oracle_requant_ex(e2m1, e4m3, scale_2, n, rows, K, 0u, codes, ue8m0);
}

/* MXFP4 tensors (reading R10): e2m1 [n][rows][K/2], UE8M0 scales [n][rows][K/32]
 * -> codes [n][rows][K/4], ue8m0 [n][rows][K/32].  Returns status bits. */
uint32_t oracle_requant_mxfp4(const uint8_t *e2m1, const uint8_t *scales, int64_t n, int64_t rows, int64_t K,
                              uint32_t options, uint8_t *codes, uint8_t *ue8m0)
{
    if (K % 32 != 0) return 0x80000000u;
    uint32_t st = 0;
    int balance = (options & ORACLE_BALANCE_ZERO_SIGNS) != 0;
    ORACLE_PARALLEL_FOR_BLOCKS
    for (int64_t g = 0; g < n * rows * (K / 32); ++g)
        st |= requant_block_mx(e2m1 + g * 16, scales[g], balance, codes + g * 8, ue8m0 + g);
    return st;
}

/* Selected blocks only (flat block index over n*rows*K/32); outputs [nb][8], [nb]. */
uint32_t oracle_requant_blocks(const uint8_t *e2m1, const uint8_t *e4m3, const float *scale_2,
                               int64_t rows, int64_t K, const int64_t *block_ids, int64_t nb,
                               uint8_t *codes, uint8_t *ue8m0)
{
    if (K % 32 != 0) return 0x80000000u;
    uint32_t st = 0;
    int64_t blocks_per_tensor = rows * (K / 32);
    ORACLE_PARALLEL_FOR_BLOCKS
    for (int64_t i = 0; i < nb; ++i) {
        int64_t g = block_ids[i];
        st |= requant_block(e2m1 + g * 16, e4m3 + g * 2, scale_2[g / blocks_per_tensor], 0,
                            codes + i * 8, ue8m0 + i);
    }
    return st;
}

/* FP8 block-quantised tensors: e4m3 bytes [n][rows][K] with one f32 scale per
 * 128 x 128 block, scales [n][ceil(rows/128)][ceil(K/128)] -> codes
 * [n][rows][K/4], ue8m0 [n][rows][K/32].  Returns status bits. */
uint32_t oracle_requant_fp8(const uint8_t *w8, const float *scales, int64_t n, int64_t rows, int64_t K,
                            uint8_t *codes, uint8_t *ue8m0)
{
    if (K % 32 != 0) return 0x80000000u;
    uint32_t st = 0;
    int64_t bpr = K / 32, srows = (rows + 127) / 128, scols = (K + 127) / 128;
    ORACLE_PARALLEL_FOR_BLOCKS
    for (int64_t g = 0; g < n * rows * bpr; ++g) {
        int64_t t = g / (rows * bpr), r = (g / bpr) % rows, b = g % bpr;
        float s = scales[(t * srows + r / 128) * scols + (b * 32) / 128];
        st |= requant_block_fp8(w8 + g * 32, s, codes + g * 8, ue8m0 + g);
    }
    return st;
}

/* ------------------------------------------------------------------ permute */

/* Stable grouping of pairs p = t*k + j by expert id: for e = 0..E-1 in order,
 * every pair of expert e in increasing p; out-of-range ids follow, in increasing
 * p.  offsets[e] = first sorted slot of expert e, offsets[E] = valid pairs. */
uint32_t oracle_permute(const int32_t *ids, int64_t T, int32_t k, int32_t E,
                        int32_t *sorted_pairs, int32_t *inv_pairs, int32_t *offsets)
{
    int64_t P = T * k, q = 0;
    uint32_t st = 0;
    for (int32_t e = 0; e < E; ++e) {
        offsets[e] = (int32_t)q;
        for (int64_t p = 0; p < P; ++p)
            if (ids[p] == e) sorted_pairs[q++] = (int32_t)p;
    }
    offsets[E] = (int32_t)q;
    for (int64_t p = 0; p < P; ++p)
        if (ids[p] < 0 || ids[p] >= E) {
            sorted_pairs[q++] = (int32_t)p;
            st |= ORACLE_BAD_EXPERT_ID;
        }
    for (int64_t i = 0; i < P; ++i) inv_pairs[sorted_pairs[i]] = (int32_t)i;
    return st;
}

/* ------------------------------------------------------------------ forward */

/* Dequantise one row of K weights: w = code_value * 2^(s-127). */
static uint32_t dequant_row(const uint8_t *codes, const uint8_t *scales, int64_t K, double *out)
{
    uint32_t st = 0;
    for (int64_t b = 0; b < K / 32; ++b) {
        unsigned s = scales[b];
        double scale = 0.0;
        if (ue8m0_valid(s)) scale = ldexp(1.0, (int)s - 127);
        else st |= ORACLE_BAD_SCALE;
        for (int64_t i = b * 32; i < b * 32 + 32; ++i) {
            unsigned c = (codes[i / 4] >> (2 * (i % 4))) & 3u;
            out[i] = oracle_code_value(c) * scale;
        }
    }
    return st;
}

/* The rows of one layer's weights, whatever their storage: fills out with row r
 * of gate/up (w13, r < 2I) or of down (w2) of slot e; returns status bits. */
typedef struct {
    uint32_t (*row)(const void *ctx, int w2, int64_t e, int64_t r, double *out);
    const void *ctx;
} RowSource;

typedef struct {
    const uint8_t *w13_codes, *w13_scales, *w2_codes, *w2_scales;
    int32_t H, I;
} Planes2;

static uint32_t row2(const void *ctx, int w2, int64_t e, int64_t r, double *out)
{
    const Planes2 *p = (const Planes2 *)ctx;
    if (!w2) {
        int64_t g = e * 2 * p->I + r;
        return dequant_row(p->w13_codes + g * (p->H / 4), p->w13_scales + g * (p->H / 32), p->H, out);
    }
    int64_t g = e * p->H + r;
    return dequant_row(p->w2_codes + g * (p->I / 4), p->w2_scales + g * (p->I / 32), p->I, out);
}

/* One NVFP4 row of K weights (reading R12): w = e2m1 * e4m3(block of 16) * s2. */
static uint32_t dequant_row_w4(const uint8_t *e2m1, const uint8_t *e4m3, double s2, int64_t K, double *out)
{
    uint32_t st = 0;
    for (int64_t b = 0; b < K / 16; ++b) {
        double sc = oracle_e4m3_value(e4m3[b]);
        if (isnan(sc)) {
            st |= ORACLE_BAD_SCALE;
            sc = 0.0;
        }
        for (int64_t i = b * 16; i < b * 16 + 16; ++i) {
            unsigned nib = (e2m1[i / 2] >> (4 * (i % 2))) & 0xFu;
            out[i] = oracle_e2m1_value(nib) * sc * s2;   /* exact: at most 2 + 4 + 24 significant bits */
        }
    }
    return st;
}

typedef struct {
    const uint8_t *w13_e2m1, *w13_e4m3, *w2_e2m1, *w2_e4m3;
    const float *w13_s2;   /* [E][2]: gate, up */
    const float *w2_s2;    /* [E] */
    int32_t H, I;
} Planes4;

static uint32_t row4(const void *ctx, int w2, int64_t e, int64_t r, double *out)
{
    const Planes4 *p = (const Planes4 *)ctx;
    if (!w2) {
        int64_t g = e * 2 * p->I + r;
        double s2 = (double)p->w13_s2[2 * e + (r < p->I ? 0 : 1)];
        return dequant_row_w4(p->w13_e2m1 + g * (p->H / 2), p->w13_e4m3 + g * (p->H / 16), s2, p->H, out);
    }
    int64_t g = e * p->H + r;
    return dequant_row_w4(p->w2_e2m1 + g * (p->I / 2), p->w2_e4m3 + g * (p->I / 16), (double)p->w2_s2[e], p->I, out);
}

static double dot(const double *a, const double *b, int64_t n)
{
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* y of token t: y_out bf16 [H]; h_out (nullable) bf16 [k][I]. */
/* Slot of a routed id under reading R9 (slot_of NULL: the id is the slot).
 * Returns the slot, -1 for a missing expert, -2 for an invalid id. */
static int32_t slot_of_pair(int32_t e, const int32_t *slot_of, int32_t n_route, int32_t S)
{
    if (slot_of) {
        if (e < 0 || e >= n_route) return -2;
        e = slot_of[e];
        if (e < 0) return -1;
    }
    return (e >= 0 && e < S) ? e : -2;
}

static uint32_t forward_token(const uint16_t *x, const int32_t *ids, const float *weights,
                              const int32_t *slot_of, int32_t n_route, const RowSource *src,
                              int32_t E, int32_t H, int32_t I, int32_t k, int64_t t,
                              uint16_t *y_out, uint16_t *h_out)
{
    uint32_t st = 0;
    double *xt = malloc(sizeof(double) * H), *row = malloc(sizeof(double) * (H > I ? H : I));
    double *h = malloc(sizeof(double) * I), *acc = malloc(sizeof(double) * H);
    if (!xt || !row || !h || !acc) oracle_fail("malloc");
    for (int32_t i = 0; i < H; ++i) xt[i] = oracle_bf16_to_double(x[t * H + i]);
    for (int32_t m = 0; m < H; ++m) acc[m] = 0.0;
    for (int32_t j = 0; j < k; ++j) {
        int32_t e = slot_of_pair(ids[t * k + j], slot_of, n_route, E);
        if (h_out)
            for (int32_t n = 0; n < I; ++n) h_out[(int64_t)j * I + n] = 0;
        if (e == -1) continue;   /* not resident: contributes nothing */
        if (e < 0) {
            st |= ORACLE_BAD_EXPERT_ID;
            continue;
        }
        double w = (double)weights[t * k + j];
        for (int32_t n = 0; n < I; ++n) {
            st |= src->row(src->ctx, 0, e, n, row);
            double g = dot(row, xt, H);
            st |= src->row(src->ctx, 0, e, (int64_t)I + n, row);
            double u = dot(row, xt, H);
            uint16_t hb = oracle_bf16_from_double(silu(g) * u);
            h[n] = oracle_bf16_to_double(hb);
            if (h_out) h_out[(int64_t)j * I + n] = hb;
        }
        for (int32_t m = 0; m < H; ++m) {
            st |= src->row(src->ctx, 1, e, m, row);
            acc[m] += w * dot(row, h, I);
        }
    }
    for (int32_t m = 0; m < H; ++m) y_out[m] = oracle_bf16_from_double(acc[m]);
    free(xt);
    free(row);
    free(h);
    free(acc);
    return st;
}

/* y for the listed tokens.  x bf16 [T][H], ids/weights [T][k]; planes as in the
 * C ABI; y_out bf16 [ntok][H]; h_out (nullable) bf16 [ntok][k][I]. */
uint32_t oracle_forward_tokens(const uint16_t *x, const int32_t *ids, const float *weights,
                               const uint8_t *w13_codes, const uint8_t *w13_scales,
                               const uint8_t *w2_codes, const uint8_t *w2_scales,
                               int32_t E, int32_t H, int32_t I, int32_t k,
                               const int64_t *tokens, int64_t ntok, uint16_t *y_out, uint16_t *h_out)
{
    if (H % 32 || I % 32) return 0x80000000u;
    Planes2 pl = {w13_codes, w13_scales, w2_codes, w2_scales, H, I};
    RowSource src = {row2, &pl};
    uint32_t st = 0;
    ORACLE_PARALLEL_FOR_TOKENS
    for (int64_t it = 0; it < ntok; ++it)
        st |= forward_token(x, ids, weights, NULL, 0, &src, E, H, I, k, tokens[it], y_out + it * H,
                            h_out ? h_out + it * k * (int64_t)I : NULL);
    return st;
}

/* The FP4 layer (reading R12): NVFP4 planes w13_e2m1 [E][2I][H/2], w13_e4m3
 * [E][2I][H/16], w13_s2 [E][2] (gate, up), w2_e2m1 [E][H][I/2], w2_e4m3
 * [E][H][I/16], w2_s2 [E]; otherwise as oracle_forward_tokens. */
uint32_t oracle_forward_tokens_w4(const uint16_t *x, const int32_t *ids, const float *weights,
                                  const uint8_t *w13_e2m1, const uint8_t *w13_e4m3, const float *w13_s2,
                                  const uint8_t *w2_e2m1, const uint8_t *w2_e4m3, const float *w2_s2,
                                  int32_t E, int32_t H, int32_t I, int32_t k,
                                  const int64_t *tokens, int64_t ntok, uint16_t *y_out, uint16_t *h_out)
{
    if (H % 32 || I % 32) return 0x80000000u;
    Planes4 pl = {w13_e2m1, w13_e4m3, w2_e2m1, w2_e4m3, w13_s2, w2_s2, H, I};
    RowSource src = {row4, &pl};
    uint32_t st = 0;
    ORACLE_PARALLEL_FOR_TOKENS
    for (int64_t it = 0; it < ntok; ++it)
        st |= forward_token(x, ids, weights, NULL, 0, &src, E, H, I, k, tokens[it], y_out + it * H,
                            h_out ? h_out + it * k * (int64_t)I : NULL);
    return st;
}

/* The same behind an expert cache (reading R9): planes of S = E slots, slot_of
 * [n_route].  *misses (nullable) = pairs of the listed tokens whose expert is
 * not resident. */
uint32_t oracle_forward_tokens_cached(const uint16_t *x, const int32_t *ids, const float *weights,
                                      const int32_t *slot_of, int32_t n_route,
                                      const uint8_t *w13_codes, const uint8_t *w13_scales,
                                      const uint8_t *w2_codes, const uint8_t *w2_scales,
                                      int32_t E, int32_t H, int32_t I, int32_t k,
                                      const int64_t *tokens, int64_t ntok, uint16_t *y_out, uint16_t *h_out,
                                      int64_t *misses)
{
    if (H % 32 || I % 32 || !slot_of) return 0x80000000u;
    Planes2 pl = {w13_codes, w13_scales, w2_codes, w2_scales, H, I};
    RowSource src = {row2, &pl};
    uint32_t st = 0;
    ORACLE_PARALLEL_FOR_TOKENS
    for (int64_t it = 0; it < ntok; ++it)
        st |= forward_token(x, ids, weights, slot_of, n_route, &src, E, H, I, k, tokens[it], y_out + it * H,
                            h_out ? h_out + it * k * (int64_t)I : NULL);
    if (misses) {
        int64_t m = 0;
        for (int64_t it = 0; it < ntok; ++it)
            for (int32_t j = 0; j < k; ++j)
                m += slot_of_pair(ids[tokens[it] * k + j], slot_of, n_route, E) == -1;
        *misses = m;
    }
    return st;
}
