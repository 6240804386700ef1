// Shared device helpers and the internal launch interface of libmoe_w2.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

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

// Decode activation operands (x for gate_up, h for down) enter the block-scaled
// MMA (e2m1 x e2m1, kind::mxf4) as kActDigits rows of packed e2m1 "digits" per
// activation row, each digit row with its own UE8M0 byte per 32 elements:
//   a = sum_r d_r * 2^(s_r - 127) + residual,
// where row r encodes, rounded to the nearest e2m1 value, what rows 0..r-1 left
// over, scaled so that the block's largest leftover maps into (3, 6].  A row
// shrinks the block's largest leftover at least threefold (about tenfold on
// typical data), so the residual is bounded relative to the block's largest
// element, not to each element.  Eight rows, measured on a CPU model of the
// rows against the oracle, reproduce x and h exactly on normal activations and
// on blocks with one element 2^8..2^12 times the others or with exact zeros
// beside large values; six rows leave up to ~2.6e-4 (relative L2 of the layer
// output) on those blocks and five ~8e-4.  Two pairs of eight rows fill the
// MMA's N = 16, so the rows beyond five cost no MMAs.
// Inside every group of 16 elements, packed position p (nibble p & 1 of byte
// p >> 1 of the row) holds element fp4_elem(p) = 2 (p & 7) + (p >> 3): the code
// expansion puts the even codes of a 16-code word in one TMEM column and the odd
// codes in the next, and the MMA reads column j nibble i as K index 8 j + i.
constexpr int kActDigits = 8;
__host__ __device__ __forceinline__ int fp4_elem(int p) { return ((p & 7) << 1) | (p >> 3); }
__host__ __device__ __forceinline__ int fp4_pos(int e) { return ((e & 1) << 3) | (e >> 1); }

// UE8M0 byte s of a digit row whose block's largest magnitude is amax: the
// smallest power of two 2^(s-127) with amax / 2^(s-127) <= 6 (so the block's
// values map into (3, 6]), within [1, 253].
__device__ __forceinline__ uint32_t digit_scale_byte(float amax)
{
    if (!(amax > 0.f)) return 127u;   // all zeros (or not a number: the values carry it)
    const uint32_t b = __float_as_uint(amax);
    const int ex = (int)((b >> 23) & 0xFFu);   // amax = m 2^(ex - 127), m in [1, 2)
    // amax / 2^(ex - 129) = 4 m <= 6 while m <= 1.5; above, one step up (2 m in (3, 4))
    const int s = ex - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
    return (uint32_t)min(253, max(1, s));
}
// 2^(s - 127) and 2^(127 - s) for s in [1, 253].
__device__ __forceinline__ float digit_scale(uint32_t s) { return __uint_as_float(s << 23); }
__device__ __forceinline__ float digit_inv_scale(uint32_t s) { return __uint_as_float((254u - s) << 23); }
// Nearest e2m1 value of v (ties to the even mantissa; |v| above 6 gives 6): the
// nibble (sign in bit 3, magnitude index of 0, .5, 1, 1.5, 2, 3, 4, 6) and its value.
__device__ __forceinline__ uint32_t e2m1_digit(float v, float& val)
{
    const float a = fminf(fabsf(v), 6.f);
    const float q = a < 2.f ? rintf(a * 2.f) * 0.5f : a < 4.f ? rintf(a) : rintf(a * 0.5f) * 2.f;
    const uint32_t mi = q < 2.f ? (uint32_t)(q * 2.f) : q < 4.f ? (uint32_t)q + 2u : q < 5.f ? 6u : 7u;
    val = v < 0.f ? -q : q;
    return mi | (v < 0.f && mi != 0u ? 8u : 0u);
}
// The same digit as e2m1_digit by the tensor-core conversion instruction:
// cvt.rn.satfinite.e2m1x2 rounds to the nearest e2m1 value (ties to the even
// mantissa) and saturates at 6; a zero keeps no sign.  Checked equal to
// e2m1_digit on every tie, the saturation edge and a million random values.
__device__ __forceinline__ uint32_t e2m1_digit_hw(float v, float& val)
{
    uint32_t n, h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(n) : "f"(0.f), "f"(v));
    n = (n & 7u) != 0u ? (n & 15u) : 0u;
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(n));
    val = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    return n;
}
// Two digits at once (lo into the low nibble, hi into the high nibble of the
// returned byte), as two e2m1_digit_hw: one conversion for both values.
__device__ __forceinline__ uint32_t e2m1x2_digits_hw(float lo, float hi, float& qlo, float& qhi)
{
    uint32_t n, h2;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}" : "=r"(n) : "f"(hi), "f"(lo));
    n &= ((n & 0x7u) != 0u ? 0x0Fu : 0u) | ((n & 0x70u) != 0u ? 0xF0u : 0u);   // a zero keeps no sign
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "r"(n));
    qlo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
    qhi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
    return n;
}

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

// ------------------------------------------------------------------ selector words (both GEMM paths)
struct SelConst {
    uint32_t m33, c04, mcc, c10, fix, k16, k4, s2, s16, s18;
};

__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t shr(uint32_t a, uint32_t n)
{
    uint32_t d;
    asm("shr.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(n));
    return d;
}
// (a & b) | c in one logic op
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Byte-permute with the selector used as is: every selector nibble built below
// has bit 3 clear, so it needs no masking (the __byte_perm intrinsic promises to
// use only 3 bits of each nibble).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}
// A value the compiler cannot see through: keeps a constant in a register, so
// every instruction below takes it as a register operand (instructions with two
// immediates would otherwise be split in two, or need a move per use).
__device__ __forceinline__ uint32_t opaque(uint32_t v)
{
    asm volatile("" : "+r"(v));
    return v;
}

// Selector words of a 16-code word w (code i in bits 2i..2i+1) for the bf16
// pairs (c_r, c_{r+4}) [lo] and (c_{r+8}, c_{r+12}) [hi].  In each selector byte
// the high nibble is the code (0..3: a byte of the lut word) and the low nibble
// is 4 | (any two bits) (a byte of the lo word); the byte-permute reads only the
// low 16 bits of a selector, so only those need to be exact.  From
//   mp  = (w & 0x33333333) | 0x04040404   codes 4b, 4b+2 of byte b, plus 4 per byte
//   m2p = (w & 0xCCCCCCCC) | 0x10101010   codes 4b+1, 4b+3, plus 0x10 per byte
// (one logic op each) the eight selectors are
//   lo: r=0 mp*16 - 0x3C3C3C3C   r=1 m2p*4 - 0x3C3C3C3C   r=2 mp   r=3 m2p >> 2
//   hi: the lo selector of the same r shifted right by 16 (r=3: m2p >> 18)
// (the subtractions remove the shifted fill and leave 0x04 per byte).  Per word:
// 2 logic ops, 5 shifts and 8 byte-permutes on the ALU pipe, 2 multiply-adds on
// the FMA pipe.  Right shifts stay shifts: as the high word of a product they
// would run on the FMA pipe at a quarter of its rate.
struct Masks {
    uint32_t mp, m2p;
};
__device__ __forceinline__ Masks word_masks(uint32_t w, const SelConst& k)
{
    return Masks{and_or(w, k.m33, k.c04), and_or(w, k.mcc, k.c10)};
}
__device__ __forceinline__ void selectors(const Masks& s, const SelConst& k, uint32_t (&lo)[4], uint32_t (&hi)[4])
{
    lo[0] = mad_lo(s.mp, k.k16, k.fix);
    lo[1] = mad_lo(s.m2p, k.k4, k.fix);
    lo[2] = s.mp;
    lo[3] = shr(s.m2p, k.s2);
    hi[0] = shr(lo[0], k.s16);
    hi[1] = shr(lo[1], k.s16);
    hi[2] = shr(s.mp, k.s16);
    hi[3] = shr(s.m2p, k.s18);
}

// The selector constants as opaque registers (loaded once per thread).
__device__ __forceinline__ SelConst sel_const_regs()
{
    SelConst k;
    k.m33 = opaque(0x33333333u);
    k.c04 = opaque(0x04040404u);
    k.mcc = opaque(0xCCCCCCCCu);
    k.c10 = opaque(0x10101010u);
    k.fix = opaque(0xC3C3C3C4u);
    k.k16 = opaque(16u);
    k.k4 = opaque(4u);
    k.s2 = opaque(2u);
    k.s16 = opaque(16u);
    k.s18 = opaque(18u);
    return k;
}

// ------------------------------------------------------------------ NVFP4 weights (the FP4 layer)
// A weight is e2m1 x e4m3 (one scale per 16 elements) x scale_2 (per tensor).
// The product e2m1 x e4m3 has at most 2 + 4 significant bits and lies in
// [2^-10, 2688], so it is exact in bf16; scale_2 multiplies the fp32
// accumulator in the epilogue.  Per scale byte s, Fp4Lut holds the bf16 high
// and low bytes of |e2m1 magnitude m| * e4m3(s) for m = 0..7 (bytes m of the
// pair (hi0, hi1) and of (lo0, lo1)), the scale's sign in the high bytes; an
// e4m3 NaN scale gives zeros (its block counts as 0).
__host__ __device__ __forceinline__ uint4 make_fp4_lut(uint32_t s)
{
    const uint32_t E = (s >> 3) & 15u, m = s & 7u;
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (E == 15u && m == 7u) return r;
    // e4m3 = (E ? 8 + m : m) * 2^((E ? E : 1) - 10); e2m1 magnitudes in halves
    const float sc = (float)(E ? 8u + m : m) * ldexpf(1.0f, (int)(E ? E : 1u) - 10) * ((s & 0x80u) ? -1.0f : 1.0f);
    const float half_units[8] = {0.f, 1.f, 2.f, 3.f, 4.f, 6.f, 8.f, 12.f};
    for (int i = 0; i < 8; ++i) {
        float v = 0.5f * half_units[i] * sc;
        uint32_t b;
        memcpy(&b, &v, 4);
        b >>= 16;   // exact: at most 6 significant bits
        const uint32_t hi = (b >> 8) & 0xFFu, lo = b & 0xFFu;
        if (i < 4) {
            r.x |= hi << (8 * i);
            r.z |= lo << (8 * i);
        } else {
            r.y |= hi << (8 * (i - 4));
            r.w |= lo << (8 * (i - 4));
        }
    }
    return r;
}
// 0x80 in every byte of w whose e4m3 value is NaN (low seven bits all ones).
__host__ __device__ __forceinline__ uint32_t e4m3_nan_bytes(uint32_t w)
{
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}
// Eight e2m1 nibbles w (byte b: element 2b low, element 2b+1 high) times their
// block's scale (table L) -> four bf16 pairs:
//   r0 = (e0, e4), r1 = (e1, e5), r2 = (e2, e6), r3 = (e3, e7)
// which is the pair order of the T16 activation layout (and of the mma.sync A
// fragments the decode kernel builds from it).  A byte-permute selector takes
// one nibble per output byte from the low 16 bits, so the bytes are first
// regrouped as (b0, b2 | b1, b3): the low half then holds the magnitudes of
// elements 0, 1, 4, 5 and the high half those of 2, 3, 6, 7.  The nibble's sign
// (bit 3 of it: bits 3, 19 of w for e0, e4; 7, 23 for e1, e5; 11, 27; 15, 31) is
// moved to bits 15 and 31 of each pair and XOR-ed into the table's sign.
__device__ __forceinline__ void fp4_word_bf16(uint32_t w, const uint4& L, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3)
{
    const uint32_t v = prmt(w, w, 0x3120u);                        // bytes b0, b2, b1, b3
    const uint32_t sa = v & 0x7777u, sb = (v >> 16) & 0x7777u;     // magnitudes (e0 e1 e4 e5), (e2 e3 e6 e7)
    const uint32_t ha = prmt(L.x, L.y, sa), la = prmt(L.z, L.w, sa);
    const uint32_t hb = prmt(L.x, L.y, sb), lb = prmt(L.z, L.w, sb);
    r0 = prmt(la, ha, 0x6240u) ^ ((w << 12) & 0x80008000u);   // e0, e4
    r1 = prmt(la, ha, 0x7351u) ^ ((w << 8) & 0x80008000u);    // e1, e5
    r2 = prmt(lb, hb, 0x6240u) ^ ((w << 4) & 0x80008000u);    // e2, e6
    r3 = prmt(lb, hb, 0x7351u) ^ (w & 0x80008000u);           // e3, e7
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

__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ------------------------------------------------------------------ workspace
// Decode split of the down projection's K for the block-scaled kernel: each
// 128-row block of W_down is cut into s_dn segments of l_dn chunks of 256, one
// work item each, so that a small step still has work for every CTA.
struct DecodeSplit {
    int32_t s_dn, l_dn;   // down: segments, chunks per segment (K = I)
};
DecodeSplit decode_split(int64_t P, int32_t E, int32_t H, int32_t I);
// Which decode kernel a step of P pairs of the 2-bit layer takes: at most 16
// pairs with H and I multiples of 512 up to 7168, the stream-K block-scaled kernel
// (decode_stream.cu); other shapes with H or I not a multiple of 512, the bf16
// mma.sync kernel (decode_mma.cu); the rest, the block-scaled kernel
// (decode.cu).  (The block-scaled kernels load weight-row scale groups by TMA,
// whose rows, H/32 and I/32 bytes, must be multiples of 16 bytes.)
bool decode_use_stream(int64_t P, int32_t H, int32_t I);
bool decode_use_mma(int64_t P, int32_t H, int32_t I);
// The stream-K decode kernel: counters it needs zeroed, and the floats of each
// of its two partial-sum buffers (one CTA per SM, at most kMaxStreamGrid).
constexpr int kMaxStreamGrid = 256;
int64_t stream_counter_count(int64_t P, int32_t H, int32_t I);
size_t stream_part_floats();   // floats of the stream-K kernel's partial sums (all phases)

struct Workspace {
    int32_t* sorted;       // [P]
    int32_t* inv;          // [P]
    int32_t* offsets;      // [E+1]
    int32_t* active;       // [E] active experts ascending
    int32_t* active_count; // [1]
    int4* tiles;           // GEMM tiles (expert, first slot, pairs, 0)
    int32_t* tile_count;   // [1]
    int32_t* counters;     // decode, zeroed by the permutation kernel.  Block-scaled kernel: per
                           // (tile, 64-row block of h) the publications of its h [max_tiles][I/64],
                           // then the item queue [1].  mma.sync kernel: see decode_counter_count
    // prefill, and the mma.sync decode kernel
    uint16_t* xa;          // activation rows, T16 layout: prefill in expert order [P][H], decode per token [T][H]
    uint16_t* h;           // SiLU(gate)*up rows in expert order, T16 layout [P][I]
    float* stage;          // per-pair outputs times router weight, slot t*k+j: prefill [P][H],
                           // decode [s_dn][P][H] (one slab per K segment of down)
    // decode
    uint8_t* xd;           // e2m1 digit rows of x, kActDigits per token [8T][H/2]
    uint8_t* sxd;          // their UE8M0 bytes [8T][H/32]
    uint8_t* hd;           // e2m1 digit rows of h, kActDigits per pair (expert order) [8P][I/2]
    uint8_t* shd;          // their UE8M0 bytes [8P][I/32]
    float* gu_part;        // block-scaled kernel: gate_up partial sums of the two K halves [2][P][2I] (small
                           // steps only, else null); stream-K kernel: the partial sums of cut row blocks,
                           // per phase (stream_part_floats() floats)
    // behind an expert cache
    int32_t* ids_eff;      // slot of each pair, -1 when left out [P] (null without a residency table)
    DecodeSplit split;
    size_t bytes;
};

Workspace carve_workspace(void* base, int32_t T, int32_t k, int32_t E, int32_t H, int32_t I, bool cached = false,
                          bool w4 = false);
int64_t max_tiles(int64_t P, int32_t E, bool decode);
int64_t decode_counter_count(int64_t P, int32_t E, int32_t H, int32_t I, bool mma);

// ------------------------------------------------------------------ launches
// Optional profiling events recorded between phases (see moe_w2_forward_traced).
// During stream capture the events become external record nodes, so each graph
// replay records them and cudaEventElapsedTime works on replays.
// One layer's expert weights as the layer kernels read them: the 2-bit planes,
// or NVFP4 experts (the FP4 layer).  2-bit: codes [rows][K/4], UE8M0 scales
// [rows][K/32].  NVFP4: e2m1 [rows][K/2], e4m3 [rows][K/16] and a per-tensor
// scale_2 (w13: [E][2], gate then up; w2: [E]).
struct LayerPlanes {
    bool w4;
    const uint8_t *w13_codes, *w13_scales, *w2_codes, *w2_scales;
    const float *w13_scale_2, *w2_scale_2;
    int32_t num_experts, hidden, inter;
};

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

// Expert residency of a step: routed id -> slot of the planes (all null: the
// routed ids are the slots).
struct PermuteSlots {
    const int32_t* slot_of = nullptr;   // [n_route], negative: not resident
    int32_t n_route = 0;
    int32_t* ids_eff = nullptr;         // [P] out: slot per pair, -1 when left out
    uint32_t* misses = nullptr;         // += pairs whose expert is not resident
};

cudaError_t launch_permute(const int32_t* ids, const PermuteSlots& slots, int32_t T, int32_t k, int32_t E,
                           int32_t* sorted, int32_t* inv, int32_t* offsets, int32_t* active, int32_t* active_count,
                           int4* tiles, int32_t* tile_count, int32_t tile_rows, const uint16_t* x, uint16_t* x_t16,
                           uint8_t* xd, uint8_t* sxd, int32_t H, int32_t* counters, int32_t n_counters, uint16_t* y,
                           uint32_t* status, cudaStream_t s);

cudaError_t launch_decode_mma(const int32_t* ids, const float* weights, const LayerPlanes& w, int32_t T, int32_t k,
                              const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                              const PhaseEvents& ev);
// ids: the pairs' experts as the permutation sorted them (cache slots behind an
// expert cache); route_ids: the routed expert ids (the tiles' canonical order);
// slot_of, n_route: the residency table behind an expert cache (else null, 0).
cudaError_t launch_decode_stream(const int32_t* ids, const int32_t* route_ids, const int32_t* slot_of,
                                 int32_t n_route, const float* weights, const moe_w2_planes& w, int32_t T, int32_t k,
                                 const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                                 const PhaseEvents& ev);
cudaError_t launch_decode(const uint16_t* x, const int32_t* ids, const float* weights,
                          const moe_w2_planes& w, int32_t T, int32_t k, const Workspace& ws, uint16_t* y,
                          uint32_t* status, cudaStream_t s, const PhaseEvents& ev);

cudaError_t launch_prefill(const uint16_t* x, const int32_t* ids, const float* weights, const LayerPlanes& w,
                           int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status,
                           cudaStream_t s, const PhaseEvents& ev);

cudaError_t launch_requant(const uint8_t* e2m1, const uint8_t* e4m3, const float* scale_2, int64_t n, int64_t rows,
                           int64_t K, uint32_t options, uint8_t* codes, uint8_t* ue8m0, uint32_t* status,
                           cudaStream_t s);
cudaError_t launch_requant_mxfp4(const uint8_t* e2m1, const uint8_t* scales, int64_t n, int64_t rows, int64_t K,
                                 uint32_t options, uint8_t* codes, uint8_t* ue8m0, uint32_t* status, cudaStream_t s);

cudaError_t launch_requant_fp8(const uint8_t* w8, const float* scales, int64_t n, int64_t rows, int64_t K,
                               uint8_t* codes, uint8_t* ue8m0, uint32_t* status, cudaStream_t s);

int sm_count();

// The cross-CTA dependency waits of the decode kernels (a down item waiting for
// the h it reads): normally a target reached by the gate_up epilogues and a limit
// of about two seconds; with the debug hook on (moe_w2_debug_force_pipeline_timeout)
// an unreachable target and a limit of about 0.1 ms, so that the wait times out.
struct DepWait {
    int32_t bias;          // added to the target
    long long limit;       // clock cycles
};
DepWait dependency_wait();
// MOE_W2_OK when the current device has compute capability 10.3, else
// MOE_W2_ERR_DEVICE (MOE_W2_ERR_CUDA if the query fails); cached per device.
moe_w2_status check_device();

// One-time set-up per device (kernel attributes, occupancy), safe under
// concurrent calls: kernel attributes belong to a device's context, so each
// device the library runs on gets its own.  `done` is the call site's table;
// init(dev) runs under one library-wide mutex until it first succeeds, and
// `dev` receives the current device.
constexpr int kMaxDevices = 64;
std::mutex& init_mutex();
template <class F>
cudaError_t once_per_device(bool (&done)[kMaxDevices], int& dev, F&& init)
{
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(init_mutex());
    if (done[dev]) return cudaSuccess;
    e = init(dev);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

}  // namespace moe_w2
