// Decode path for the smallest steps (at most 16 pairs): every active expert's
// 2-bit planes streamed from HBM once per layer by a stream-K split over one
// CTA per SM, multiplied on the tensor cores in block-scaled FP4
// (tcgen05.mma kind::mxf4), with the weighted combine in the same launch.
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": codes expanded in
// registers and fed to block-scaled tensor-core MMAs; section "FP4 recovery":
// decode is HBM-bound, the 2-bit read is the cost.  Page "The v0.24.0 port",
// section "Benchmarks": tokens grouped by expert, so each active expert's
// weights are read once per step however many tokens use it; "Deterministic
// unpermute" bullet: per-pair results are placed in their own slot and summed
// over top_k in a fixed order.
//
// The operands are those of the block-scaled kernel of decode.cu: a weight is
// +-1 or +-4 under its row's UE8M0 byte of a 32-element block, i.e. an e2m1
// value under an MX block scale; the code expansion is one nibble per code
// ((c << 2) | 2); activations (x, then h) enter as kActDigits rows of e2m1
// digits each, 8 of the MMA's N = 32 columns per pair, four pairs per tile.
//
// Work split (stream-K).  A row block is 128 weight rows of one tile: gate_up
// the 64 gate rows of a 64-element block of h with its 64 up rows (K = H),
// down 128 rows of W_down (K = I); a chunk is 256 K of a row block.  The chunks
// of all gate_up row blocks (tile-major) form one sequence and those of all
// down row blocks another; CTA b takes the b-th of gridDim.x equal ranges of
// each, so every SM streams the same number of plane bytes.  A row block cut by
// range boundaries is summed from fp32 partials, by whichever of its CTAs
// arrives last, in range order (a fixed order: the result does not depend on
// which CTA finishes first).  The partial of a range is kept in one of two
// slots: 0 for the row block the range starts in, 1 for the one it ends in.
// Gate_up epilogues publish h of their 64 elements as digit rows; a down chunk
// waits (bounded) until the four h blocks of its K range are published.  Down
// epilogues write w * (W_down h) into the pair's fp32 slot; the last of a 128-row
// block of y's n_tiles contributions sums every token's slots in j order into y.
// The waits assume the grid's CTAs are co-resident (one per SM, sized to the
// SM count): a wait that cannot end gives up with the pipeline-timeout status.
//
// Roles (sixteen warps, one CTA per SM):
//   warps 0-3   consumers, one per TMEM lane quadrant, one thread per weight row:
//               expand the row's 256 codes of a chunk to packed e2m1 and store
//               them with the row's two scale words and the activation rows'
//               scale words into the chunk's A stage in TMEM
//   warps 4-7   epilogues (one per TMEM lane quadrant): read each run's
//               accumulators, hand them back, then finish their 32 rows
//   warps 8-11  code producers, one pair of chunks in four each: stream the
//               pair's code tile (128 rows x 128 bytes, 128B-swizzled) by TMA
//               into an 8-slot ring, running ahead of the consumers (down chunks
//               included: their codes do not wait for h); lane 1 of warp 8 sends
//               every run's scale tile (the 128 rows' whole scale rows) into one
//               of two buffers
//   warps 12-13 activation producers, one pair of chunks in two each: per pair
//               of the tile its digit rows (two 8 x 128-byte boxes, 128B-swizzled
//               as the UMMA B operand) and their scale group by TMA into a
//               4-slot ring; down chunks only once the h of their tiles is
//               published
//   warps 14-15 MMA issuers (one thread each): issuer q takes the chunks of a run
//               with index q mod 2, four MMAs (M = 128, N = 32, K = 64) per chunk
//               into its own accumulator of the run's set; four sets rotate over
//               consecutive runs, so the MMAs run up to three row blocks ahead of
//               the slowest epilogue
// (A single thread issues one tensor copy every few hundred cycles whatever its
// size, and one chunk's MMAs and commits in about as long: hence six producers
// and two issuers.)
#include <algorithm>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kChunk = 256;                          // K per chunk: 4 MMAs of K = 64
constexpr int kRows = 128;                           // weight rows per row block (MMA M)
constexpr int kTilePairs = 4;                        // pairs per tile
constexpr int kN = 32;                               // MMA N: the digit rows of a tile's pairs
static_assert(kActDigits * kTilePairs <= kN, "a tile's digit rows must fit the MMA N");
constexpr int kCWarps = 4;                           // consumer warps 0-3
constexpr int kEpiWarp0 = 4;                         // epilogue warps 4-7 (TMEM lane quadrants 0-3)
constexpr int kEWarps = 4;
constexpr int kCodeWarp0 = 8;                        // code producers: warps 8-11
constexpr int kCodeWarps = 4;
constexpr int kActWarp0 = 12;                        // activation producers: warps 12-13
constexpr int kActWarps = 2;
constexpr int kMmaWarp0 = 14;                        // MMA issuers: warps 14-15
constexpr int kIssuers = 2;
constexpr int kThreads = 16 * 32;
constexpr int kAccSets = 4;                          // accumulator sets: runs g use set g % 4
constexpr int kCSlots = 8;                           // code ring (pair-chunk tiles)
constexpr int kBSlots = 4;                           // activation ring (pair-chunk tiles)
constexpr int kStages = 5;                           // A stages in TMEM (one chunk each)
constexpr uint32_t kCodeBytes = kRows * 128;         // a pair of chunks: 128 rows x 128 code bytes, 128B-swizzled
constexpr uint32_t kBTile = 8 * 128;                 // one pair's 8 digit rows of one chunk (a 128B swizzle atom)
constexpr uint32_t kBSfOff = 2 * kTilePairs * kBTile;   // in a B slot: tiles (pair j, chunk h) at (2 j + h) kBTile,
constexpr uint32_t kBSlotBytes = kBSfOff + 1024;        // then pair j's 8 x 16 scale bytes at kBSfOff + 128 j
constexpr uint32_t kOffB = kCSlots * kCodeBytes;     // activation slots (1024-aligned)
constexpr uint32_t kOffS = kOffB + kBSlots * kBSlotBytes;   // two scale tiles of 128 rows x sb bytes
static_assert(kCodeBytes % 1024 == 0 && kOffB % 1024 == 0 && kBSlotBytes % 1024 == 0,
              "swizzled tiles need 1024-byte alignment");
// every ring slot has a single producer (pair position s goes to producer s mod n)
static_assert(kCSlots % kCodeWarps == 0 && kBSlots % kActWarps == 0, "producers own whole slots");
constexpr int kMaxScaleRow = 224;                    // scale bytes of a row (H/32, I/32): H, I <= 7168
constexpr uint32_t kTmemCols = 512;
// accumulator of set s, issuer q: columns 32 (2 s + q); A stage st: 256 + 32 st;
// scale words: A (stage st, word w, lane quadrant q) 416 + 8 st + 4 w + q, B
// (stage st, word w) 456 + 8 st + 4 w (scale operands start on 4-column boundaries)
constexpr uint32_t kColA = 256;
constexpr uint32_t kColSfa = 416;
constexpr uint32_t kColSfb = 456;
static_assert(32 * kIssuers * kAccSets <= kColA && kColA + 32 * kStages <= kColSfa &&
                  kColSfa + 8 * kStages <= kColSfb && kColSfb + 8 * kStages <= kTmemCols,
              "TMEM layout");
// Sleeps between polls of the warps that wait most of the time (a warp spinning
// on a barrier takes issue slots from the consumer warp of its sub-partition)
constexpr uint32_t kProducerSleepNs = 64;
constexpr uint32_t kEpiSleepNs = 100;
constexpr uint32_t kIssuerSleepNs = 20;
constexpr int32_t kHPublished = 2;                   // release adds per 64-element block of h (one per 32)
constexpr int kMaxStreamTiles = 32;                  // tiles of a step (at most one per pair)

struct StreamArgs {
    int32_t H, I, T, k, E;
    int64_t P;
    const int4* tiles;
    const int32_t* tile_count;
    const int32_t* sorted;
    const float* weights;
    const int32_t* ids;          // [T][k]: kept pairs (valid ids) for the final sum
    const int32_t* route_ids;    // [T][k]: routed expert ids (the order of the tiles' row blocks)
    const int32_t* slot_of;      // behind an expert cache: [n_route] slot of each routed id (else null)
    int32_t n_route;
    uint8_t* hd;                 // [8P][I/2] digit rows of h
    uint8_t* shd;                // [8P][I/32]
    float* stage;                // [P][H] w * (W_down h) per pair
    float* part_g;               // [grid][2][kTilePairs][128] gate_up partial sums
    float* part_d;               // [grid][2][kTilePairs][128] down partial sums
    int32_t* h_flag;             // [tiles][I/64] h publications (one per 32 elements)
    int32_t* g_cnt;              // [tiles][I/64][2] gate_up partials arrived, per 32 elements of h
    int32_t* d_cnt;              // [tiles][H/128][4] down partials arrived, per 32 rows
    int32_t* y_cnt;              // [H/128][4] tiles done with 32 rows of y
    uint16_t* y;
    int32_t sb;                  // bytes per row of a scale tile (max(H, I) / 32)
    DepWait dep;
    uint32_t* status;
};

// A tile of the step as the producers and epilogues read it.
struct TileInfo {
    int q0, nrows;               // first slot of the sorted pairs, pairs
    int pr[kTilePairs];          // its pairs (t * k + j)
    int tok[kTilePairs];         // their tokens
    float w[kTilePairs];         // their router weights
};

struct SharedState {
    uint64_t full_c[kCSlots];    // code producers -> consumers: a pair of chunks' code tile landed
    uint64_t empty_c[kCSlots];   // consumer warps -> code producer: slot read
    uint64_t full_s[2];          // code producers -> consumers: a run's scale tile landed
    uint64_t empty_s[2];         // consumer warps -> code producer: scale tile read
    uint64_t full_b[kBSlots];    // activation producers -> consumers, issuers: digit rows landed
    uint64_t empty_b[kBSlots];   // both issuers' commits -> activation producer: slot read
    uint64_t a_full[kStages];    // consumer warps -> issuer: A stage written
    uint64_t a_empty[kStages];   // MMA commit -> consumers: A stage read
    uint64_t d_full[kAccSets];   // both issuers' commits -> epilogue warps: accumulator set complete
    uint64_t d_empty[kAccSets];  // epilogue warps -> issuers: accumulator set read
    uint64_t u_full[2][2];       // up-row warp 2 + h -> gate-row warp h: up sums in u_box (per half h, slot)
    uint64_t u_free[2][2];       // gate-row warp h -> up-row warp 2 + h: u_box slot read
    uint64_t drain;
    uint64_t tiles_ready;        // warp 0 -> activation producers, epilogue warps: tinfo written
    TileInfo tinfo[kMaxStreamTiles];   // by row-block position (routed-id order)
    int plane_of[kMaxStreamTiles];     // planes' expert index of each tile position
    int n_tiles;
    float u_box[2][2][kTilePairs][32];   // up-row sums of whole gate_up row blocks (half, slot)
    uint32_t tmem;
    int abort_flag;
};

// Shared-memory descriptor of a K-major operand in the 128-byte swizzle layout
// (as smem_desc_sw128) whose 8-row groups lie sbo bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128_sbo(uint32_t saddr, uint32_t sbo)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ int32_t ld_acquire_s32(const int32_t* p)
{
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Add with release semantics at GPU scope: this thread's earlier writes, and
// those it has observed (the warp's, after __syncwarp), are visible to a thread
// that reads the new value with an acquire.
__device__ __forceinline__ void red_release_add(int32_t* p, int32_t v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int32_t atom_add_acq_rel(int32_t* p, int32_t v)
{
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Orders this thread's view of global memory (h another CTA wrote with plain
// stores and published, acquired here) before its later tensor copies of it.
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Two words of packed e2m1 from one word of 16 codes: nibble n of r0 holds code
// 2n and nibble n of r1 code 2n + 1, each as (c << 2) | 2 (c in bits 3:2: +1,
// +4, -1, -4).  One shift and two and-or operations per word.
__device__ __forceinline__ void expand_fp4(uint32_t w, uint32_t& r0, uint32_t& r1)
{
    asm("{\n\t.reg .b32 t0;\n\t"
        "shl.b32 t0, %2, 2;\n\t"
        "lop3.b32 %0, t0, 0xCCCCCCCC, 0x22222222, 0xEA;\n\t"   // (x & m) | c
        "lop3.b32 %1, %2, 0xCCCCCCCC, 0x22222222, 0xEA;\n\t}"
        : "=r"(r0), "=r"(r1)
        : "r"(w));
}

// Nonzero when a byte of the scale word s is outside [1, 252] (may also flag a
// valid byte above an invalid one; the caller re-checks byte by byte).
__device__ __forceinline__ uint32_t scale_word_suspect(uint32_t s)
{
    const uint32_t d = s - 0x01010101u;
    return ((d & 0x7F7F7F7Fu) + 0x04040404u) & d & 0x80808080u;
}

// Scale words of a chunk with every byte outside [1, 252] replaced by 127 (a
// unit scale), and the mask of those bytes (bit t: byte t % 4 of word t / 4,
// the scale of the chunk's 32-element block t).  Out of line: it runs only for
// invalid planes, and the consumers' loop stays small.
struct ScaleFix {
    uint32_t x, y, mask;
};
static __device__ __noinline__ ScaleFix fix_scale_words(uint32_t x, uint32_t y)
{
    ScaleFix f{x, y, 0u};
    for (int t = 0; t < 8; ++t) {
        uint32_t& wv = t < 4 ? f.x : f.y;
        const int sh8 = 8 * (t & 3);
        if (((wv >> sh8) & 0xFFu) - 1u > 251u) {
            wv = (wv & ~(0xFFu << sh8)) | (127u << sh8);
            f.mask |= 1u << t;
        }
    }
    return f;
}

// A pair's accumulator row: the sum of its kActDigits digit columns.
__device__ __forceinline__ float pair_sum(const float (&v)[32], int j)
{
    float s = 0.f;
#pragma unroll
    for (int d = 0; d < kActDigits; ++d) s += v[kActDigits * j + d];
    return s;
}

// h of one 32-element block and one pair (one value per lane, block element =
// lane) as kActDigits digit rows of pair slot q: the lane's element sits at
// packed position pos of the block; the other nibble of its byte belongs to
// lane ^ 2, and the lane with the low nibble writes the byte.
__device__ __forceinline__ void store_h_digits(const StreamArgs& a, int64_t q, int blk, float v)
{
    const int lane = threadIdx.x & 31;
    const int pos = (lane & 16) | fp4_pos(lane & 15);
#pragma unroll
    for (int d = 0; d < kActDigits; ++d) {
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const uint32_t sd = digit_scale_byte(__uint_as_float(amax_bits));
        float qv;
        const uint32_t nib = e2m1_digit(v * digit_inv_scale(sd), qv);
        v -= qv * digit_scale(sd);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 2);
        const int64_t row = kActDigits * q + d;
        if ((pos & 1) == 0) a.hd[row * (a.I / 2) + blk * 16 + (pos >> 1)] = (uint8_t)(nib | (other << 4));
        if (lane == 0) a.shd[row * (a.I / 32) + blk] = (uint8_t)sd;
    }
}

// One of the two chunk sequences (gate_up or down) cut into nr equal ranges of
// whole chunk pairs (the unit the code tiles come in; a row block holds an even
// number of chunks), nr = min(grid, pairs) so that no range is empty (CTAs
// b >= nr get none).  Chunk indices throughout.
struct Seq {
    int64_t n;    // chunks
    int32_t L;    // chunks per row block
    int32_t nr;   // ranges
    __device__ __forceinline__ Seq(int64_t n_, int32_t L_, int32_t grid)
        : n(n_), L(L_), nr((int32_t)(n_ / 2 < (int64_t)grid ? n_ / 2 : (int64_t)grid)) {}
    __device__ __forceinline__ int64_t start(int64_t b) const { return b < nr ? 2 * (b * (n / 2) / nr) : n; }
    // the range holding chunk i (the last range starting at or before its pair)
    __device__ __forceinline__ int64_t range_of(int64_t i) const { return ((i / 2 + 1) * nr - 1) / (n / 2); }
};

// A CTA's walk over its chunks: its gate_up range, then its down range.  Every
// role steps through the same positions in order (next()), and keeps the index
// g of the current run (consecutive chunks of one row block) and the position j
// of the chunk in it.
struct Walk {
    int64_t g0, ng, d0, nd;    // range starts and lengths
    int32_t Lg, Ld;
    int p = -1, g = -1, j = 0;
    int kind = 0;              // 1 gate_up, 0 down
    int64_t R = 0;             // row block (tile-major within its sequence)
    int c = 0;                 // chunk of the row block
    bool first = false, last = false;
    __device__ __forceinline__ int total() const { return (int)(ng + nd); }
    __device__ __forceinline__ void next()
    {
        ++p;
        if (p < ng) {
            if (p == 0) {
                kind = 1;
                R = g0 / Lg;
                c = (int)(g0 % Lg);
            } else if (++c == Lg) {
                c = 0;
                ++R;
            }
            first = p == 0 || c == 0;
            last = p == ng - 1 || c == Lg - 1;
        } else {
            if (p == ng) {
                kind = 0;
                R = d0 / Ld;
                c = (int)(d0 % Ld);
            } else if (++c == Ld) {
                c = 0;
                ++R;
            }
            first = p == ng || c == 0;
            last = p == ng + nd - 1 || c == Ld - 1;
        }
        if (first) {
            ++g;
            j = 0;
        } else {
            ++j;
        }
    }
};

// A run (a row block's chunks inside this CTA's range) as the epilogue needs it.
struct Run {
    int kind;
    int64_t R;
    int g;          // run index (accumulator set g % kAccSets)
    int nchunks;    // chunks of the run (1: only issuer 0's accumulator was written)
};

// Epilogue of run `r` by one epilogue warp (TMEM lane quadrant qd = warp % 4,
// rows m = 32 qd + lane); the four warps work on their own, so that each
// finishes its 32 rows (or 32 elements of h) without waiting for the others:
//   gate_up  the 32 elements 64 rb + 32 h + lane of h (h = qd % 2) need gate row
//            32 h + lane (warp h) and up row 64 + 32 h + lane (warp 2 + h).  The
//            whole row block in this CTA: the up warp hands its sums to the
//            gate warp (shared memory, two slots); cut by ranges: both write
//            their range's part slot and count in, and the warp whose count
//            completes the 2 x parts (in any CTA) sums the parts in range order.
//            Then h = bf16(SiLU(gate) * up) as digit rows, published by one
//            release add per 32 elements.
//   down     the warp's 32 rows: directly (whole row block) or, when cut, by the
//            warp whose count completes the row block's parts; w * (W_down h)
//            into the pairs' slots, then one count for these rows of y; the
//            count that completes them (n_tiles) sums every token's slots of
//            the 32 rows in j order into y.
// wn: whole gate_up runs so far of this warp (the u_box slot sequence).
__device__ __noinline__ void epilogue(const StreamArgs& a, SharedState& sh, uint32_t tq, const Run& r,
                                      const Seq& sg, const Seq& sd, int n_tiles, int wn, volatile int* abort)
{
    const int lane = threadIdx.x & 31, qd = (threadIdx.x >> 5) & 3, m = 32 * qd + lane;
    const uint32_t set = (uint32_t)r.g % kAccSets;
    const bool ok = mbar_wait_warp(smem_u32(&sh.d_full[set]), ((uint32_t)r.g / kAccSets) & 1u, abort, kEpiSleepNs);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    if (ok) {
        tc_fence_after();
        tmem_ld32(tq + 32u * (2u * set), v);
        if (r.nchunks > 1) {
            float v1[32];
            tmem_ld32(tq + 32u * (2u * set + 1u), v1);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += v1[i];
        }
        tc_fence_before();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.d_empty[set]));
    if (!ok) return;

    const bool gate_up = r.kind == 1;
    const Seq& sq = gate_up ? sg : sd;
    const int rbn = gate_up ? a.I / 64 : a.H / 128;   // row blocks per tile
    const int ti = (int)(r.R / rbn), rb = (int)(r.R % rbn);
    const TileInfo& tile = sh.tinfo[ti];
    const int nrows = tile.nrows;
    // the ranges rf..rl cut the row block; the part slot of range rg
    const int64_t rf = sq.range_of(r.R * sq.L), rl = sq.range_of((r.R + 1) * sq.L - 1);
    const int nparts = (int)(rl - rf + 1);
    float s[kTilePairs];
#pragma unroll
    for (int j = 0; j < kTilePairs; ++j) s[j] = pair_sum(v, j);
    float* part = gate_up ? a.part_g : a.part_d;
    auto part_ptr = [&](int64_t rg, int j, int row) {
        const int slot = (r.R == sq.start(rg) / sq.L) ? 0 : 1;
        return part + (((rg * 2 + slot) * kTilePairs + j) * kRows + row);
    };
    // the row block's sum of pair j, row `row` over its parts in range order
    // (loads four at a time, so their latencies overlap)
    auto total = [&](int j, int row) {
        float t = 0.f;
        int64_t rg = rf;
        for (; rg + 3 <= rl; rg += 4) {
            const float x0 = __ldcg(part_ptr(rg, j, row)), x1 = __ldcg(part_ptr(rg + 1, j, row));
            const float x2 = __ldcg(part_ptr(rg + 2, j, row)), x3 = __ldcg(part_ptr(rg + 3, j, row));
            t += x0;
            t += x1;
            t += x2;
            t += x3;
        }
        for (; rg <= rl; ++rg) t += __ldcg(part_ptr(rg, j, row));
        return t;
    };
    int old = 0;

    if (gate_up) {
        const int h = qd & 1;   // the 32 elements 64 rb + 32 h + lane of h
        float g[kTilePairs], u[kTilePairs];
        if (nparts == 1) {
            const int slot = wn & 1;
            const uint32_t ph = ((uint32_t)wn >> 1) & 1u;
            if (qd >= 2) {
                // up rows: hand the sums to the gate warp of this half
                if (!mbar_wait_warp(smem_u32(&sh.u_free[h][slot]), ph ^ 1u, abort, kEpiSleepNs)) return;
#pragma unroll
                for (int j = 0; j < kTilePairs; ++j) sh.u_box[h][slot][j][lane] = s[j];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.u_full[h][slot]));
                return;
            }
            if (!mbar_wait_warp(smem_u32(&sh.u_full[h][slot]), ph, abort, kEpiSleepNs)) return;
#pragma unroll
            for (int j = 0; j < kTilePairs; ++j) {
                g[j] = s[j];
                u[j] = sh.u_box[h][slot][j][lane];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.u_free[h][slot]));
        } else {
            for (int j = 0; j < nrows; ++j) *part_ptr(blockIdx.x, j, m) = s[j];
            __syncwarp();   // the warp's stores come before lane 0's release
            if (lane == 0) old = atom_add_acq_rel(a.g_cnt + 2 * r.R + h, 1);
            if (__shfl_sync(0xffffffffu, old, 0) != 2 * nparts - 1) return;
            __syncwarp();   // the lanes' reads below come after lane 0's acquire
            for (int j = 0; j < nrows; ++j) {
                g[j] = total(j, 32 * h + lane);
                u[j] = total(j, 64 + 32 * h + lane);
            }
        }
        for (int j = 0; j < nrows; ++j) {
            const float hv = __bfloat162float(__float2bfloat16_rn(silu_f(g[j]) * u[j]));
            store_h_digits(a, (int64_t)tile.q0 + j, 2 * rb + h, hv);
        }
        __syncwarp();
        if (lane == 0) red_release_add(a.h_flag + r.R, 1);
        return;
    }

    // down: this warp's 32 rows into the pairs' slots
    const int row = kRows * rb + m;
    if (nparts > 1) {
        for (int j = 0; j < nrows; ++j) *part_ptr(blockIdx.x, j, m) = s[j];
        __syncwarp();
        if (lane == 0) old = atom_add_acq_rel(a.d_cnt + 4 * r.R + qd, 1);
        if (__shfl_sync(0xffffffffu, old, 0) != nparts - 1) return;
        __syncwarp();
        for (int j = 0; j < nrows; ++j) s[j] = total(j, m);
    }
    for (int j = 0; j < nrows; ++j) a.stage[(int64_t)tile.pr[j] * a.H + row] = tile.w[j] * s[j];
    __syncwarp();   // the warp's stores come before lane 0's release
    if (lane == 0) old = atom_add_acq_rel(a.y_cnt + 4 * rb + qd, 1);
    if (__shfl_sync(0xffffffffu, old, 0) != n_tiles - 1) return;
    __syncwarp();
    // every tile's slots of these 32 rows are written: y = their sum per token
    // in j order (pairs left out never wrote a slot and add nothing)
    for (int t = 0; t < a.T; ++t) {
        float acc = 0.f;
        for (int j = 0; j < a.k; ++j) {
            const int e = __ldg(a.ids + t * a.k + j);
            if ((unsigned)e < (unsigned)a.E) acc += __ldcg(a.stage + (int64_t)(t * a.k + j) * a.H + row);
        }
        __nv_bfloat16 yb = __float2bfloat16_rn(acc);
        a.y[(int64_t)t * a.H + row] = *reinterpret_cast<uint16_t*>(&yb);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
decode_stream_kernel(const __grid_constant__ CUtensorMap gu_map, const __grid_constant__ CUtensorMap dn_map,
                     const __grid_constant__ CUtensorMap gu_sf_map, const __grid_constant__ CUtensorMap dn_sf_map,
                     const __grid_constant__ CUtensorMap xd_map, const __grid_constant__ CUtensorMap sxd_map,
                     const __grid_constant__ CUtensorMap hd_map, const __grid_constant__ CUtensorMap shd_map,
                     const StreamArgs a)
{
    __shared__ SharedState sh;
    extern __shared__ uint8_t dyn_smem[];   // kOffS + 2 * 128 * sb + 1024 (aligned below)
    const uint32_t ring_addr = (smem_u32(dyn_smem) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kCSlots; ++s) {
            mbar_init(smem_u32(&sh.full_c[s]), 1);
            mbar_init(smem_u32(&sh.empty_c[s]), kCWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sh.full_s[s]), 1);
            mbar_init(smem_u32(&sh.empty_s[s]), kCWarps);
        }
        for (int s = 0; s < kBSlots; ++s) {
            mbar_init(smem_u32(&sh.full_b[s]), 1);
            mbar_init(smem_u32(&sh.empty_b[s]), kIssuers);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.a_full[s]), kCWarps);
            mbar_init(smem_u32(&sh.a_empty[s]), 1);
        }
        for (int s = 0; s < kAccSets; ++s) {
            mbar_init(smem_u32(&sh.d_full[s]), kIssuers);
            mbar_init(smem_u32(&sh.d_empty[s]), kEWarps);
        }
        for (int h = 0; h < 2; ++h)
            for (int s = 0; s < 2; ++s) {
                mbar_init(smem_u32(&sh.u_full[h][s]), 1);
                mbar_init(smem_u32(&sh.u_free[h][s]), 1);
            }
        mbar_init(smem_u32(&sh.drain), kIssuers);
        mbar_init(smem_u32(&sh.tiles_ready), 1);
        sh.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh.tmem), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kCodeWarp0 && lane == 0) {
        prefetch_tmap(&gu_map);
        prefetch_tmap(&dn_map);
        prefetch_tmap(&gu_sf_map);
        prefetch_tmap(&dn_sf_map);
    }
    if (warp == kActWarp0 && lane == 0) {
        prefetch_tmap(&xd_map);
        prefetch_tmap(&sxd_map);
        prefetch_tmap(&hd_map);
        prefetch_tmap(&shd_map);
    }
    if (warp == 1) {
        // The step's tiles in the order of their routed expert ids, from the
        // routing itself (an input: no need to wait for the permutation kernel),
        // so the code producers can start at once: each kept expert (ascending
        // routed id) gets ceil(pairs / 4) tiles, as the permutation forms them.
        // Behind an expert cache the planes' index of expert r is its slot.
        // At most 32 pairs (one per lane).
        int r = -1, plane = -1;
        if (lane < a.P) {
            r = __ldg(a.route_ids + lane);
            if (a.slot_of != nullptr) plane = (unsigned)r < (unsigned)a.n_route ? __ldg(a.slot_of + r) : -1;
            else plane = r;
            if ((unsigned)plane >= (unsigned)a.E) r = -1;
        }
        const int key = r >= 0 ? r : 0x7FFFFFFF;
        const uint32_t same = __match_any_sync(0xffffffffu, key);
        const bool lead = r >= 0 && (__ffs(same) - 1) == lane;
        const int ntl = lead ? (__popc(same) + kTilePairs - 1) / kTilePairs : 0;
        int before = 0, total = 0;
        for (int u = 0; u < 32; ++u) {
            const int ku = __shfl_sync(0xffffffffu, key, u), nu = __shfl_sync(0xffffffffu, ntl, u);
            before += ku < key ? nu : 0;
            total += nu;
        }
        for (int t = 0; t < ntl; ++t) sh.plane_of[before + t] = plane;
        if (lane == 0) sh.n_tiles = total;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh.tmem;
    volatile int* abort = &sh.abort_flag;
    const int n_tiles = sh.n_tiles;
    const int rbg = a.I / 64, rbd = a.H / 128;
    const Seq sg((int64_t)n_tiles * rbg * (a.H / kChunk), a.H / kChunk, (int32_t)gridDim.x);
    const Seq sd((int64_t)n_tiles * rbd * (a.I / kChunk), a.I / kChunk, (int32_t)gridDim.x);
    Walk w0{};
    w0.g0 = sg.start(blockIdx.x);
    w0.ng = sg.start(blockIdx.x + 1) - w0.g0;
    w0.d0 = sd.start(blockIdx.x);
    w0.nd = sd.start(blockIdx.x + 1) - w0.d0;
    w0.Lg = sg.L;
    w0.Ld = sd.L;
    const int total = w0.total();   // even: ranges hold whole chunk pairs
    const uint32_t sbuf0 = ring_addr + kOffS;
    const uint32_t sbytes = (uint32_t)kRows * (uint32_t)a.sb;   // one scale tile

    if (warp >= kCodeWarp0 && warp < kCodeWarp0 + kCodeWarps) {
        // ------------------------------------------------ code producers (read only inputs)
        // Lane 0 of producer w issues the pairs of chunks s = w mod kCodeWarps
        // (one pair: 128 rows x 128 code bytes in one tensor copy); a single
        // thread issues one tensor copy every few hundred cycles, so one
        // producer could not keep the ring full.  Lane 1 of producer 0 issues
        // every run's scale tile (every weight row's whole scale row in one
        // copy), in run order: a buffer's next tile is then sent only once the
        // tile before it was both sent and read, so no wait on the buffer can
        // mistake an older phase for the one it waits for.
        const int w = warp - kCodeWarp0;
        if (lane == 0) {
            Walk wk = w0;
            int p = 0;
            for (; p < total; ++p) {
                wk.next();
                const int sp = p >> 1;
                if ((p & 1) || sp % kCodeWarps != w) continue;
                const bool gu = wk.kind == 1;
                const int rb = (int)(wk.R % (gu ? rbg : rbd));
                const int e = sh.plane_of[wk.R / (gu ? rbg : rbd)];
                const uint32_t slot = (uint32_t)sp % kCSlots;
                if (!mbar_wait_sleep(smem_u32(&sh.empty_c[slot]), (((uint32_t)sp / kCSlots) & 1u) ^ 1u, abort,
                                     kProducerSleepNs))
                    break;
                const uint32_t base = ring_addr + slot * kCodeBytes, fb = smem_u32(&sh.full_c[slot]);
                mbar_arrive_expect_tx_relaxed(fb, kCodeBytes);
                // chunks c, c + 1 of the row block: code bytes 64 c .. 64 c + 127 of every row
                if (gu) {
                    // 64 gate rows then their 64 up rows (planes 2e, 2e + 1 of the
                    // w13 plane seen as 2E planes of I rows)
                    tma_load_3d(base, &gu_map, wk.c * 64, 64 * rb, 2 * e, fb);
                } else {
                    tma_load_2d(base, &dn_map, wk.c * 64, e * a.H + kRows * rb, fb);
                }
            }
            if (*abort) {
                // the consumers may have stopped before the last tiles landed: wait
                // (bounded) for this producer's copies of the last ring positions
                volatile int never = 0;
                const int sp_end = (p + 1) >> 1;
                for (int sq = sp_end > kCSlots ? sp_end - kCSlots : 0; sq < sp_end; ++sq)
                    if (sq % kCodeWarps == w)
                        (void)mbar_wait(smem_u32(&sh.full_c[sq % kCSlots]), ((uint32_t)sq / kCSlots) & 1u, &never);
            }
        } else if (lane == 1 && w == 0) {
            // the run's scale tile into buffer g % 2, once run g - 2 is done with it
            Walk wk = w0;
            int last_g[2] = {-1, -1};   // the last run whose tile went to each buffer
            for (int p = 0; p < total; ++p) {
                wk.next();
                if (!wk.first) continue;
                const bool gu = wk.kind == 1;
                const int rb = (int)(wk.R % (gu ? rbg : rbd));
                const int e = sh.plane_of[wk.R / (gu ? rbg : rbd)];
                const uint32_t b = (uint32_t)wk.g & 1u;
                if (!mbar_wait_sleep(smem_u32(&sh.empty_s[b]), (((uint32_t)wk.g >> 1) & 1u) ^ 1u, abort,
                                     kProducerSleepNs))
                    break;
                const uint32_t fs = smem_u32(&sh.full_s[b]);
                mbar_arrive_expect_tx_relaxed(fs, kRows * (uint32_t)(gu ? a.H / 32 : a.I / 32));
                if (gu) tma_load_3d(sbuf0 + b * sbytes, &gu_sf_map, 0, 64 * rb, 2 * e, fs);
                else tma_load_2d(sbuf0 + b * sbytes, &dn_sf_map, 0, e * a.H + kRows * rb, fs);
                last_g[b] = wk.g;
            }
            if (*abort) {
                volatile int never = 0;
                for (int b = 0; b < 2; ++b)
                    if (last_g[b] >= 0)
                        (void)mbar_wait(smem_u32(&sh.full_s[b]), ((uint32_t)last_g[b] >> 1) & 1u, &never);
            }
        }
    } else {
        // Launched as a programmatic dependent of the permutation kernel:
        // everything it writes (tiles, zeroed counters, x digits) is read only
        // after this wait.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (warp == 0) {
            // the tiles' pairs (the permutation's tile list, put in the order
            // above): first slot, pairs, their tokens and router weights
            int key = 0;
            int4 t4 = make_int4(0, 0, 0, 0);
            if (lane < n_tiles) {
                t4 = a.tiles[lane];
                key = a.slot_of != nullptr ? __ldg(a.route_ids + __ldg(a.sorted + t4.y)) : t4.x;
            }
            int rank = 0;
            for (int u = 0; u < n_tiles; ++u) {
                const int ku = __shfl_sync(0xffffffffu, key, u);
                rank += (ku < key || (ku == key && u < lane)) ? 1 : 0;
            }
            if (lane < n_tiles) {
                TileInfo& ti = sh.tinfo[rank];
                ti.q0 = t4.y;
                ti.nrows = t4.z;
                for (int j = 0; j < kTilePairs; ++j) {
                    const int pr = j < t4.z ? __ldg(a.sorted + t4.y + j) : 0;
                    ti.pr[j] = pr;
                    ti.tok[j] = pr / a.k;
                    ti.w[j] = j < t4.z ? __ldg(a.weights + pr) : 0.f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.tiles_ready));
        }
        const bool tiles_ok = mbar_wait_warp(smem_u32(&sh.tiles_ready), 0u, abort, kProducerSleepNs);
        if (warp >= kActWarp0 && warp < kActWarp0 + kActWarps) {
            // ------------------------------------------------ activation producers
            // (producer w issues the pairs of chunks s = w mod kActWarps: per pair
            // of the tile, two digit-row boxes and one scale box)
            const int w = warp - kActWarp0;
            Walk wk = w0;
            int p = 0;
            bool waited_h = false;
            for (; p < total && tiles_ok; ++p) {
                wk.next();
                const int sp = p >> 1;
                if ((p & 1) || sp % kActWarps != w) continue;
                const uint32_t slot = (uint32_t)sp % kBSlots;
                int ok = 1;
                if (lane == 0)
                    ok = mbar_wait_sleep(smem_u32(&sh.empty_b[slot]), (((uint32_t)sp / kBSlots) & 1u) ^ 1u, abort,
                                         kProducerSleepNs);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (wk.kind == 0 && !waited_h) {
                    // the down range reads h of every tile it touches: wait
                    // (bounded) until all of those 64-element blocks are published
                    waited_h = true;
                    const int t0 = (int)(wk.d0 / wk.Ld / rbd), t1 = (int)((wk.d0 + wk.nd - 1) / wk.Ld / rbd);
                    const int nf = (t1 - t0 + 1) * rbg;
                    const int32_t* hf = a.h_flag + (int64_t)t0 * rbg;
                    const int32_t target = kHPublished + a.dep.bias;
                    auto all_ready = [&]() {
                        bool r = true;
                        for (int i = lane; i < nf; i += 32) r = r && ld_acquire_s32(hf + i) >= target;
                        return __all_sync(0xffffffffu, r);
                    };
                    if (!all_ready()) {
                        const long long c0 = clock64();
                        bool timed_out = false;
                        while (!all_ready()) {
                            if (__shfl_sync(0xffffffffu, *abort, 0)) break;
                            if (clock64() - c0 > a.dep.limit) {
                                timed_out = true;
                                break;
                            }
                            __nanosleep(128);
                        }
                        if (timed_out && lane == 0) *abort = 1;
                    }
                    __syncwarp();
                    if (__shfl_sync(0xffffffffu, *abort, 0)) break;
                    fence_proxy_async_global();
                }
                const TileInfo& tile = sh.tinfo[wk.R / (wk.kind == 1 ? rbg : rbd)];
                const uint32_t fb = smem_u32(&sh.full_b[slot]);
                if (lane == 0)
                    mbar_arrive_expect_tx_relaxed(fb, (uint32_t)tile.nrows * (kActDigits * (2 * 128 + 16)));
                __syncwarp();
                if (lane < tile.nrows) {
                    // pair `lane` of the tile: gate_up reads its token's rows of x, down its rows of h
                    const int brow = kActDigits * (wk.kind == 1 ? tile.tok[lane] : tile.q0 + lane);
                    const uint32_t base = ring_addr + kOffB + slot * kBSlotBytes;
                    const CUtensorMap* dm = wk.kind == 1 ? &xd_map : &hd_map;
                    tma_load_2d(base + (2 * lane) * kBTile, dm, wk.c * 128, brow, fb);
                    tma_load_2d(base + (2 * lane + 1) * kBTile, dm, (wk.c + 1) * 128, brow, fb);
                    tma_load_2d(base + kBSfOff + lane * (kActDigits * 16), wk.kind == 1 ? &sxd_map : &shd_map,
                                wk.c * 8, brow, fb);
                }
            }
            if (*abort && lane == 0) {
                volatile int never = 0;
                const int sp_end = (p + 1) >> 1;
                for (int sq = sp_end > kBSlots ? sp_end - kBSlots : 0; sq < sp_end; ++sq)
                    if (sq % kActWarps == w)
                        (void)mbar_wait(smem_u32(&sh.full_b[sq % kBSlots]), ((uint32_t)sq / kBSlots) & 1u, &never);
            }
        } else if (warp >= kMmaWarp0) {
            // ------------------------------------------------ MMA issuers
            // Runs start on even positions, so issuer q takes the chunks p = q mod 2
            // (its own accumulator of the run's set); each also commits the B
            // slot it read, which is free once both chunks of the pair are done.
            const int q = warp - kMmaWarp0;
            if (lane == 0) {
                Walk wk = w0;
                for (int p = 0; p < total; ++p) {
                    wk.next();
                    const uint32_t set = (uint32_t)wk.g % kAccSets;
                    // The accumulator set of run g is free once the epilogue of run
                    // g - kAccSets read it.  Both issuers wait at every run's start:
                    // d_full[set] takes one commit from each, so neither may commit
                    // for a later run of the set before the epilogue of this one
                    // has seen both of its commits.
                    if (wk.first && wk.g >= kAccSets &&
                        !mbar_wait_sleep(smem_u32(&sh.d_empty[set]), (((uint32_t)wk.g / kAccSets) - 1u) & 1u, abort,
                                         kIssuerSleepNs))
                        break;
                    if ((p & 1) == q) {
                        const uint32_t st = (uint32_t)p % kStages, sp = (uint32_t)p >> 1, bs = sp % kBSlots;
                        if (!mbar_wait_sleep(smem_u32(&sh.full_b[bs]), (sp / kBSlots) & 1u, abort, kIssuerSleepNs) ||
                            !mbar_wait_sleep(smem_u32(&sh.a_full[st]), ((uint32_t)p / kStages) & 1u, abort,
                                             kIssuerSleepNs))
                            break;
                        tc_fence_after();
                        // this chunk's B tiles: pair j at (2 j + q) kBTile of the slot
                        const uint64_t bd =
                            smem_desc_sw128_sbo(ring_addr + kOffB + bs * kBSlotBytes + (uint32_t)q * kBTile, 2 * kBTile);
                        const uint32_t d = tm + 32u * (2u * set + (uint32_t)q);
                        // MMA t: K 64t..64t+63 of the chunk = A columns 8t..8t+7 of the
                        // stage, 32 bytes of every B row, scale word t / 2, bytes
                        // 2 (t % 2) and 2 (t % 2) + 1
#pragma unroll
                        for (uint32_t t = 0; t < 4; ++t)
                            umma_mxf4_ts(d, tm + kColA + 32 * st + 8 * t, bd + 2 * t,
                                         idesc_mxf4(kRows, kN, 2 * (t & 1), 2 * (t & 1)),
                                         tm + kColSfa + 8 * st + 4 * (t >> 1), tm + kColSfb + 8 * st + 4 * (t >> 1),
                                         (wk.j >= 2 || t != 0) ? 1u : 0u);
                        umma_commit(smem_u32(&sh.a_empty[st]));
                        umma_commit(smem_u32(&sh.empty_b[bs]));
                    }
                    if (wk.last) umma_commit(smem_u32(&sh.d_full[set]));
                }
                // every MMA of both issuers has completed before tensor memory is freed
                umma_commit(smem_u32(&sh.drain));
                volatile int never = 0;
                (void)mbar_wait(smem_u32(&sh.drain), 0u, &never);
            }
        } else if (warp >= kEpiWarp0) {
            // ------------------------------------------------ epilogue warps
            const uint32_t tq = tm + ((uint32_t)(32 * (warp & 3)) << 16);
            Walk wk = w0;
            int run_start = 0, wn = 0;
            for (int p = 0; p < total; ++p) {
                wk.next();
                if (wk.first) run_start = p;
                if (wk.last) {
                    epilogue(a, sh, tq, Run{wk.kind, wk.R, wk.g, p - run_start + 1}, sg, sd, n_tiles, wn, abort);
                    // whole gate_up row blocks use the u_box slots in turn
                    if (wk.kind == 1 && sg.range_of(wk.R * sg.L) == sg.range_of((wk.R + 1) * sg.L - 1)) ++wn;
                }
            }
        } else {
            // ------------------------------------------------ consumers
            const int m = tid;   // weight row of the row block
            const uint32_t tq = tm + ((uint32_t)(32 * warp) << 16);
            const uint32_t swz = (uint32_t)m & 7u;   // 128B swizzle of this code row
            uint32_t bad_scale = 0;
            Walk wk = w0;
            for (int p = 0; p < total; ++p) {
                wk.next();
                const uint32_t sp = (uint32_t)p >> 1, half = (uint32_t)p & 1u;
                const uint32_t cs = sp % kCSlots, st = (uint32_t)p % kStages, bs = sp % kBSlots;
                const uint32_t sb_run = (uint32_t)wk.g & 1u;
                bool got = true;
                if (wk.first) got = mbar_wait(smem_u32(&sh.full_s[sb_run]), ((uint32_t)wk.g >> 1) & 1u, abort);
                got = got && mbar_wait2(smem_u32(&sh.full_c[cs]), (sp / kCSlots) & 1u, smem_u32(&sh.a_empty[st]),
                                        (((uint32_t)p / kStages) & 1u) ^ 1u, abort);
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
                // the row's 64 code bytes of this chunk (16-byte unit 4 half + u of
                // the 128-byte row at (4 half + u) ^ swz) and its two scale words
                const uint32_t sb = ring_addr + cs * kCodeBytes + m * 128;
                uint32_t wd[16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 v = lds_u4(sb + (((4u * half + (uint32_t)u) ^ swz) << 4));
                    wd[4 * u] = v.x;
                    wd[4 * u + 1] = v.y;
                    wd[4 * u + 2] = v.z;
                    wd[4 * u + 3] = v.w;
                }
                uint2 sfa = lds_u2(sbuf0 + sb_run * sbytes + (uint32_t)m * (uint32_t)(wk.kind == 1 ? a.H / 32 : a.I / 32) +
                                   8u * (uint32_t)wk.c);
                __syncwarp();
                if (lane == 0) {
                    if (half) mbar_arrive(smem_u32(&sh.empty_c[cs]));   // both chunks of the pair read
                    if (wk.last) mbar_arrive(smem_u32(&sh.empty_s[sb_run]));
                }
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) expand_fp4(wd[i], r[2 * i], r[2 * i + 1]);
                if (scale_word_suspect(sfa.x) | scale_word_suspect(sfa.y)) {
                    // an invalid scale byte: that 32-element block (4 registers) counts as zero
                    const ScaleFix f = fix_scale_words(sfa.x, sfa.y);
                    sfa = make_uint2(f.x, f.y);
                    if (f.mask) {
                        bad_scale = 1;
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = ((f.mask >> (i >> 2)) & 1u) ? 0u : r[i];
                    }
                }
                // the digit rows' scale words (this quadrant's copy) come with the rows:
                // B row n's 16-byte group of the chunk pair at kBSfOff + 16 n
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.full_b[bs]), (sp / kBSlots) & 1u, abort))) break;
                const uint2 sfb = lds_u2(ring_addr + kOffB + bs * kBSlotBytes + kBSfOff + (lane % kN) * 16 + 8u * half);
                tmem_st_stage4(tq + kColA + 32 * st, r, tq + kColSfa + 8 * st + warp, sfa.x,
                               tq + kColSfa + 8 * st + 4 + warp, sfa.y, tq + kColSfb + 8 * st, sfb.x,
                               tq + kColSfb + 8 * st + 4, sfb.y);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.a_full[st]));
            }
            if (bad_scale) flag_status(a.status, MOE_W2_DEV_BAD_SCALE);
        }
    }

    tc_fence_before();
    cta_barrier_all_threads();   // every thread done before tensor memory is freed
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
    if (tid == 0 && *abort) flag_status(a.status, kDevPipelineTimeout);
}

}  // namespace

int64_t stream_counter_count(int64_t P, int32_t H, int32_t I)
{
    // per tile (at most one per pair): h publications per 64-element block of h,
    // gate_up arrivals per 32 elements of h, down arrivals per 32 rows of W_down;
    // then the tiles done per 32 rows of y
    return P * (3 * (I / 64) + 4 * (H / 128)) + 4 * (H / 128);
}

size_t stream_part_floats() { return (size_t)kMaxStreamGrid * 2 * kTilePairs * kRows; }

cudaError_t launch_decode_stream(const int32_t* ids, const int32_t* route_ids, const int32_t* slot_of,
                                 int32_t n_route, const float* weights, const moe_w2_planes& w, int32_t T, int32_t k,
                                 const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                                 const PhaseEvents& ev)
{
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    if (P > kMaxStreamTiles || std::max(H, I) / 32 > kMaxScaleRow) return cudaErrorInvalidValue;
    const int32_t sb = std::max(H, I) / 32;
    const int dyn = (int)(kOffS + 2u * kRows * (uint32_t)sb + 1024u);
    constexpr int kDynMax = (int)(kOffS + 2u * kRows * kMaxScaleRow + 1024u);
    static bool ready[kMaxDevices];
    int dev = 0;
    cudaError_t e = once_per_device(ready, dev, [&](int) -> cudaError_t {
        cudaError_t r = cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynMax);
        if (r != cudaSuccess) return r;
        return cudaFuncSetAttribute(decode_stream_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;

    StreamArgs a{};
    a.H = H;
    a.I = I;
    a.T = T;
    a.k = k;
    a.E = E;
    a.P = P;
    a.tiles = ws.tiles;
    a.tile_count = ws.tile_count;
    a.sorted = ws.sorted;
    a.weights = weights;
    a.ids = ids;
    a.route_ids = route_ids;
    a.slot_of = slot_of;
    a.n_route = n_route;
    a.hd = ws.hd;
    a.shd = ws.shd;
    a.stage = ws.stage;
    a.part_g = ws.gu_part;
    a.part_d = ws.gu_part + stream_part_floats();
    // counters, zeroed by the permutation kernel: [P][I/64] h flags, [P][I/64][2]
    // gate_up arrivals, [P][H/128][4] down arrivals, [H/128][4] y quarter blocks
    a.h_flag = ws.counters;
    a.g_cnt = a.h_flag + P * (I / 64);
    a.d_cnt = a.g_cnt + 2 * P * (I / 64);
    a.y_cnt = a.d_cnt + 4 * P * (H / 128);
    a.y = y;
    a.sb = sb;
    a.dep = dependency_wait();
    a.status = status;

    // code tiles of a pair of chunks: 128 bytes (512 codes) x 128 rows,
    // 128B-swizzled; gate_up as a 3-D box {128 bytes, 64 rows, 2 planes} over the
    // w13 plane seen as 2E planes (gate, up) of I rows, down as a 2-D box of 128 rows
    CUtensorMap gu_map, dn_map;
    if ((e = make_tmap_3d_u8(&gu_map, w.w13_codes, 2 * (int64_t)E, I, H / 4, 128, 64, 2, 128)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&dn_map, w.w2_codes, false, (int64_t)E * H, I / 4, 128, 128, 128)) != cudaSuccess) return e;
    // scale tiles of a run: every weight row's whole scale row (H/32 or I/32
    // bytes, multiples of 16 for H, I multiples of 512) x 64 rows x 2 planes
    // (gate_up) or x 128 rows (down)
    CUtensorMap gu_sf_map, dn_sf_map;
    if ((e = make_tmap_3d_u8(&gu_sf_map, w.w13_scales, 2 * (int64_t)E, I, H / 32, H / 32, 64, 2, 0)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&dn_sf_map, w.w2_scales, false, (int64_t)E * H, I / 32, I / 32, 128, 0)) != cudaSuccess)
        return e;
    // activation digit rows: boxes of one pair's 8 rows x 128 bytes (256 K),
    // 128B-swizzled as the UMMA B operand, and their 16-byte scale groups (two chunks)
    CUtensorMap xd_map, sxd_map, hd_map, shd_map;
    if ((e = make_tmap_2d(&xd_map, ws.xd, false, (int64_t)kActDigits * T, H / 2, 128, kActDigits, 128)) != cudaSuccess ||
        (e = make_tmap_2d(&sxd_map, ws.sxd, false, (int64_t)kActDigits * T, H / 32, 16, kActDigits, 0)) != cudaSuccess ||
        (e = make_tmap_2d(&hd_map, ws.hd, false, (int64_t)kActDigits * P, I / 2, 128, kActDigits, 128)) != cudaSuccess ||
        (e = make_tmap_2d(&shd_map, ws.shd, false, (int64_t)kActDigits * P, I / 32, 16, kActDigits, 0)) != cudaSuccess)
        return e;

    const int grid = std::min(sm_count(), (int)kMaxStreamGrid);
    if ((e = ev.record(1, s)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // may start before the permutation ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, decode_stream_kernel, gu_map, dn_map, gu_sf_map, dn_sf_map, xd_map, sxd_map,
                                hd_map, shd_map, a)) != cudaSuccess)
        return e;
    return ev.record(2, s);   // y is summed inside the kernel: phase 3 is empty
}

}  // namespace moe_w2
