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
// Roles (twenty warps, one CTA per SM):
//   warps 0-7   consumers in two groups (group h: warps 4h..4h+3, one per TMEM
//               lane quadrant, one thread per weight row) taking chunk h of
//               every pair: expand the row's 256 codes to packed e2m1 and store
//               them with the row's two scale words and the activation rows'
//               scale words into one of the group's two A stages in TMEM
//   warps 8-15  epilogues in two sets of four (one warp per TMEM lane quadrant),
//               set e taking the runs g with g % 2 = e: read the run's
//               accumulators, hand them back, then finish their 32 rows
//   warp 16     lane 0 streams every pair's code tile (128 rows x 128 bytes,
//               128B-swizzled) by TMA into an 8-slot ring, running ahead of the
//               consumers (down pairs included: their codes do not wait for h);
//               lane 1 sends every run's scale tile (the 128 rows' whole scale
//               rows) into one of two buffers
//   warp 17     activation producer: per pair of the tile its digit rows of
//               both chunks (one 8 x 128-byte x 2-chunk box, 128B-swizzled as
//               the UMMA B operand) and their scale group by TMA into a ring
//               sized for the step's largest tile (4 to 10 slots); down pairs
//               only once the h of their tiles is published
//   warps 18-19 MMA issuers (one thread each): issuer q takes the chunks of
//               group q, four MMAs (M = 128, N = 32, K = 64) per chunk into its
//               own accumulator of the run's set; four sets rotate over
//               consecutive runs, so the MMAs run up to three row blocks ahead
//               of the slowest epilogue
// (A consumer's chunk is a chain of dependent steps, barrier polls, shared
// loads, integer expansion at half rate, a TMEM store: two groups overlap two
// chains per quadrant.)
#include <algorithm>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kChunk = 256;                          // K per chunk: 4 MMAs of K = 64
constexpr int kRows = 128;                           // weight rows per row block (MMA M)
constexpr int kTilePairs = 4;                        // pairs per tile
constexpr int kN = 32;                               // MMA N: the digit rows of a tile's pairs
static_assert(kActDigits * kTilePairs <= kN, "a tile's digit rows must fit the MMA N");
constexpr int kGroups = 2;                           // consumer groups: group h takes chunk h of every pair
constexpr int kCWarps = 8;                           // consumer warps 0-7 (group h: warps 4h..4h+3)
constexpr int kEpiWarp0 = 8;                         // epilogue warps 8-15: two sets (runs g, g % 2 = set) of four
constexpr int kEWarps = 4;                           // warps of a set (TMEM lane quadrants 0-3)
constexpr int kESets = 2;
constexpr int kProdWarp = 16;                        // lane 0: code tiles, lane 1: scale tiles
constexpr int kActWarp = 17;                         // activation producer
constexpr int kMmaWarp0 = 18;                        // MMA issuers: warps 18-19 (issuer q feeds on group q)
constexpr int kIssuers = kGroups;
constexpr int kThreads = 20 * 32;
constexpr int kAccSets = 4;                          // accumulator sets: runs g use set g % 4
constexpr int kCSlots = 8;                           // code ring (pair tiles)
constexpr int kBSlotsMax = 12;                       // activation ring (pair tiles), sized per step
constexpr int kGStages = 2;                          // A stages in TMEM per group (one chunk each)
constexpr uint32_t kCodeBytes = kRows * 128;         // a pair of chunks: 128 rows x 128 code bytes, 128B-swizzled
constexpr uint32_t kBTile = 8 * 128;                 // one pair's 8 digit rows of one chunk (a 128B swizzle atom)
constexpr uint32_t kBRegion = 35 * 1024;             // the activation ring's bytes (4 slots of a 4-pair tile)
constexpr uint32_t kOffB = kCSlots * kCodeBytes;     // activation slots (1024-aligned)
constexpr uint32_t kOffS = kOffB + kBRegion;         // two scale tiles of 128 rows x sb bytes
static_assert(kCodeBytes % 1024 == 0 && kOffB % 1024 == 0, "swizzled tiles need 1024-byte alignment");
constexpr int kMaxScaleRow = 224;                    // scale bytes of a row (H/32, I/32): H, I <= 7168
constexpr uint32_t kTmemCols = 512;
// accumulator of set s, issuer q: columns 32 (2 s + q); A stage st (group h's
// stage i is st = 2 h + i): 256 + 32 st; scale words: A (stage st, word w, lane
// quadrant q) 384 + 8 st + 4 w + q, B (stage st, word w) 416 + 8 st + 4 w (scale
// operands start on 4-column boundaries)
constexpr int kStages = kGroups * kGStages;
constexpr uint32_t kColA = 256;
constexpr uint32_t kColSfa = 384;
constexpr uint32_t kColSfb = 416;
static_assert(32 * kIssuers * kAccSets <= kColA && kColA + 32 * kStages <= kColSfa &&
                  kColSfa + 8 * kStages <= kColSfb && kColSfb + 8 * kStages <= kTmemCols,
              "TMEM layout");
// Sleeps between polls of the warps that wait most of the time (a warp spinning
// on a barrier takes issue slots from the consumer warp of its sub-partition)
constexpr uint32_t kProducerSleepNs = 64;
constexpr uint32_t kEpiSleepNs = 100;
constexpr uint32_t kIssuerSleepNs = 20;
constexpr uint32_t kConsumerSleepNs = 32;
constexpr int32_t kHPublished = 2;                   // release adds per 64-element block of h (one per 32)
constexpr int kMaxStreamTiles = 32;                  // tiles of a step (at most one per pair)

struct StreamArgs {
    int32_t H, I, T, k, E;
    int64_t P;
    const float* weights;        // [T][k] router weights
    const int32_t* ids;          // [T][k]: kept pairs (valid ids) for the final sum
    const int32_t* route_ids;    // [T][k]: routed expert ids (the order of the tiles' row blocks)
    const int32_t* slot_of;      // behind an expert cache: [n_route] slot of each routed id (else null)
    int32_t n_route;
    uint8_t* hd;                 // [8P][I/2] digit rows of h
    uint8_t* shd;                // [8P][I/32]
    float* stage;                // [P][H] w * (W_down h) per pair
    float* part;                 // [phase][grid][2][kTilePairs][128] partial sums of cut row blocks
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

// The step's work in phases, each a chunk sequence cut into gridDim.x ranges
// (Seq below): gate_up of each tile group, then down of each tile group; a CTA
// streams its range of each in that order.  With kTileGroups = 2 the first
// group's h would be published while the second group's gate_up streams; it
// measured slower than one group (44.7 against 43.7 us for 8 pairs, 62.1
// against 60.1 for 16: every run adds an epilogue and a cut), so the tiles form
// one group.  Row blocks keep their step-wide index (tile-major per projection)
// for the counters; the cuts and part slots are per phase.
constexpr int kTileGroups = 1;
constexpr int kPhases = 2 * kTileGroups;
struct PhaseTable {
    int32_t start[kPhases], len[kPhases];   // this CTA's range of each phase (chunks of the phase)
    int32_t n[kPhases];                      // chunks of each phase
    int32_t rbase[kPhases];                  // row block (step-wide) of each phase's first
    int32_t t0[kPhases];                     // first tile of each phase
};
constexpr size_t kPartPhaseFloats = (size_t)kMaxStreamGrid * 2 * kTilePairs * kRows;

struct SharedState {
    uint64_t full_c[kCSlots];    // code producer -> consumers: a pair of chunks' code tile landed
    uint64_t empty_c[kCSlots];   // the eight consumer warps -> code producer: slot read
    uint64_t full_s[2];          // scale producer -> consumers: a run's scale tile landed
    uint64_t empty_s[2];         // the eight consumer warps -> scale producer: scale tile read
    uint64_t full_b[kBSlotsMax]; // activation producers -> consumers, issuers: digit rows landed
    uint64_t empty_b[kBSlotsMax];   // both issuers' commits -> activation producer: slot read
    uint64_t a_full[kStages];    // a group's four warps -> its issuer: A stage written
    uint64_t a_empty[kStages];   // the issuer's commit -> its group: A stage read
    uint64_t d_full[kAccSets];   // both issuers' commits -> epilogue warps: accumulator set complete
    uint64_t d_empty[kAccSets];  // epilogue warps -> issuers: accumulator set read
    uint64_t u_full[kESets][2][2];   // up-row warp 2 + h -> gate-row warp h of a set: up sums in u_box (half, slot)
    uint64_t u_free[kESets][2][2];   // gate-row warp h -> up-row warp 2 + h: u_box slot read
    uint64_t drain;
    TileInfo tinfo[kMaxStreamTiles];   // by row-block position (routed-id order)
    int plane_of[kMaxStreamTiles];     // planes' expert index of each tile position
    int n_tiles;
    int nmax;                          // pairs of the step's largest tile
    PhaseTable pt;                     // this CTA's ranges of the four phases
    float w_of[32];                    // router weight of each pair
    float u_box[kESets][2][2][kTilePairs][32];   // up-row sums of whole gate_up row blocks (set, half, slot)
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

// Element j of a register array of kTilePairs values (selects, so that a
// run-time j keeps the array in registers).
__device__ __forceinline__ float pick(const float (&v)[kTilePairs], int j)
{
    float r = v[0];
#pragma unroll
    for (int i = 1; i < kTilePairs; ++i) r = j == i ? v[i] : r;
    return r;
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
// (Rolled loops here and in the epilogue: the epilogue runs a few times per
// launch, each time mostly from cold instruction caches, so its code is kept
// small rather than unrolled.)
__device__ __forceinline__ void store_h_digits(const StreamArgs& a, int64_t q, int blk, float v)
{
    const int lane = threadIdx.x & 31;
    const int pos = (lane & 16) | fp4_pos(lane & 15);
    const int hs = a.I / 2, ss = a.I / 32;   // bytes per digit row, per scale row
    uint8_t* hp = a.hd + kActDigits * q * hs + blk * 16 + (pos >> 1);
    uint8_t* sp = a.shd + kActDigits * q * ss + blk;
#pragma unroll 1
    for (int d = 0; d < kActDigits; ++d, hp += hs, sp += ss) {
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const uint32_t sd = digit_scale_byte(__uint_as_float(amax_bits));
        float qv;
        const uint32_t nib = e2m1_digit_hw(v * digit_inv_scale(sd), qv);
        v -= qv * digit_scale(sd);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 2);
        if ((pos & 1) == 0) *hp = (uint8_t)(nib | (other << 4));
        if (lane == 0) *sp = (uint8_t)sd;
    }
}

// The sum of pair j, row `row` of a row block over its parts rf..rl in range
// order (slot 0 but for range rf, whose slot is slot_rf; loads four at a time,
// so their latencies overlap).
__device__ __noinline__ float part_total(const float* part, int rf, int rl, int slot_rf, int j, int row)
{
    auto ptr = [&](int rg) {
        return part + (((int64_t)(rg * 2 + (rg == rf ? slot_rf : 0)) * kTilePairs + j) * kRows + row);
    };
    float t = 0.f;
    int rg = rf;
    for (; rg + 3 <= rl; rg += 4) {
        const float x0 = __ldcg(ptr(rg)), x1 = __ldcg(ptr(rg + 1)), x2 = __ldcg(ptr(rg + 2)), x3 = __ldcg(ptr(rg + 3));
        t += x0;
        t += x1;
        t += x2;
        t += x3;
    }
    for (; rg <= rl; ++rg) t += __ldcg(ptr(rg));
    return t;
}

// One of the two chunk sequences (gate_up or down) cut into nr equal ranges of
// whole chunk pairs (the unit the code tiles come in; a row block holds an even
// number of chunks), nr = min(grid, pairs) so that no range is empty (CTAs
// b >= nr get none).  Chunk indices throughout.
// (32-bit: a step has at most 32 tiles x 112 row blocks x 28 chunks, and the
// products below stay under 2^24.)
struct Seq {
    int32_t n;    // chunks
    int32_t L;    // chunks per row block
    int32_t nr;   // ranges
    __device__ __forceinline__ Seq(int32_t n_, int32_t L_, int32_t grid)
        : n(n_), L(L_), nr(n_ / 2 < grid ? n_ / 2 : grid) {}
    __device__ __forceinline__ int32_t start(int32_t b) const { return b < nr ? 2 * (b * (n / 2) / nr) : n; }
    // the range holding chunk i (the last range starting at or before its pair)
    __device__ __forceinline__ int32_t range_of(int32_t i) const { return ((i / 2 + 1) * nr - 1) / (n / 2); }
};

// A CTA's runs, phase after phase, each phase's range cut at row block ends.  A
// run is the chunks of one row block inside the range, always whole pairs
// (ranges hold whole pairs and row blocks an even number of chunks).  In each
// range the row blocks cut by its ends come first and the whole ones after: a
// cut row block's other part belongs to the neighbouring CTA, which also takes
// it first, so both parts are done early, and the range's last epilogue (the
// one the next phase or y waits for) needs no other CTA.  Every role steps
// through the same runs in order (next()).
struct RunIter {
    const PhaseTable* pt;
    int32_t Lg, Ld;            // chunks per row block
    int g = -1;                // run index (accumulator set g % kAccSets, scale buffer g % 2)
    int ph = 0;                // phase
    int k = -1;                // run of the current phase's range
    int kind = 1;              // 1 gate_up, 0 down
    int32_t Rl = 0;            // row block within the phase
    int32_t R = 0;             // row block, step-wide (tile-major within its projection)
    int c0 = 0;                // first chunk of the run in the row block (even)
    int npairs = 0;            // pairs of the run
    // run kk of the range [s, s + n) of a phase with row blocks of L chunks: the
    // row blocks cut by the range's ends first, then the whole ones
    __device__ __forceinline__ bool range_run(int32_t s, int32_t n, int32_t L, int kk)
    {
        if (n <= 0) return false;
        const int32_t e = s + n, Rs = s / L, Re = (e - 1) / L;
        int32_t lo, hi;
        if (Rs == Re) {
            if (kk > 0) return false;
            Rl = Rs;
            lo = s;
            hi = e;
        } else {
            const bool hc = s != Rs * L, tc = e != (Re + 1) * L;   // head, tail row block cut
            const int ncut = (hc ? 1 : 0) + (tc ? 1 : 0);
            if (kk < ncut) {
                Rl = (kk == 0 && hc) ? Rs : Re;
                lo = Rl == Rs ? s : Re * L;
                hi = Rl == Rs ? (Rs + 1) * L : e;
            } else {
                Rl = Rs + (hc ? 1 : 0) + (kk - ncut);
                if (Rl > Re - (tc ? 1 : 0)) return false;
                lo = Rl * L;
                hi = lo + L;
            }
        }
        c0 = lo - Rl * L;
        npairs = (hi - lo) / 2;
        return true;
    }
    __device__ __forceinline__ bool next()
    {
        ++k;
        while (ph < kPhases) {
            kind = ph < kTileGroups ? 1 : 0;
            if (range_run(pt->start[ph], pt->len[ph], kind ? Lg : Ld, k)) {
                ++g;
                R = pt->rbase[ph] + Rl;
                return true;
            }
            ++ph;
            k = 0;
        }
        return false;
    }
};

// The activation ring: slots of `stride` bytes in the kBRegion bytes at kOffB,
// sized for the step's largest tile (nmax pairs) so that small tiles get a deep
// ring: pair j's digit tile of chunk h at (2 j + h) kBTile of a slot, its 8 x 16
// scale bytes at sfoff + 128 j.  The MMA reads B rows of all four pair groups
// (kBWindow bytes from the slot start, past a small slot into the next), so the
// slots are as many as keep that window of the last one inside the region (at
// most kBSlotsMax).  Every role keeps its own position (slot, phase of its
// barriers), advanced per pair.
constexpr uint32_t kBWindow = 2 * kTilePairs * kBTile;
static_assert(kBRegion >= kBWindow, "the MMA's B window fits the ring");
struct BRing {
    uint32_t stride, sfoff, nb;
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ explicit BRing(int nmax)
        : stride(((uint32_t)nmax * (2 * kBTile + 8 * 16) + 1023u) & ~1023u),
          sfoff((uint32_t)nmax * 2 * kBTile),
          nb(1u + (kBRegion - kBWindow) / stride < (uint32_t)kBSlotsMax ? 1u + (kBRegion - kBWindow) / stride
                                                                          : (uint32_t)kBSlotsMax)
    {
    }
    __device__ __forceinline__ void advance()
    {
        if (++slot == nb) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// A run (a row block's chunks inside this CTA's range) as the epilogue needs it.
struct Run {
    int kind;
    int32_t R;      // row block, step-wide
    int g;          // run index (accumulator set g % kAccSets)
    int ph;         // phase
    int32_t Rl;     // row block within the phase
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
// wn: whole gate_up runs so far of this warp's set (the u_box slot sequence).
__device__ __forceinline__ void epilogue(const StreamArgs& a, SharedState& sh, uint32_t tq, const Run r, int n_tiles,
                                         int wn, volatile int* abort)
{
    const int lane = threadIdx.x & 31, qd = (threadIdx.x >> 5) & 3, m = 32 * qd + lane;
    const int es = ((threadIdx.x >> 5) - kEpiWarp0) / kEWarps;   // epilogue set
    const uint32_t set = (uint32_t)r.g % kAccSets;
    const bool ok = mbar_wait_warp(smem_u32(&sh.d_full[set]), ((uint32_t)r.g / kAccSets) & 1u, abort, kEpiSleepNs);
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    if (ok) {
        tc_fence_after();
        // both issuers wrote their accumulator (a run has at least one pair:
        // one chunk of each group)
        float v1[32];
        tmem_ld32(tq + 32u * (2u * set), v);
        tmem_ld32(tq + 32u * (2u * set + 1u), v1);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += v1[i];
        tc_fence_before();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.d_empty[set]));
    if (!ok) return;

    const bool gate_up = r.kind == 1;
    const Seq sq(sh.pt.n[r.ph], gate_up ? a.H / kChunk : a.I / kChunk, (int32_t)gridDim.x);
    const int rbn = gate_up ? a.I / 64 : a.H / 128;   // row blocks per tile
    const int ti = (int)(r.R / rbn), rb = (int)(r.R % rbn);
    const TileInfo& tile = sh.tinfo[ti];
    const int nrows = tile.nrows;
    // the ranges rf..rl cut the row block.  A range keeps its part of the row
    // block it starts in in slot 0 and of the one it ends in in slot 1: only the
    // first range, rf, can start before this row block (slot 1 unless it starts
    // exactly at the row block's first chunk), the others start inside it.
    const int rf = sq.range_of(r.Rl * sq.L), rl = sq.range_of((r.Rl + 1) * sq.L - 1);
    const int nparts = rl - rf + 1;
    const int slot_rf = sq.start(rf) < r.Rl * sq.L ? 1 : 0;
    float s[kTilePairs];
#pragma unroll
    for (int j = 0; j < kTilePairs; ++j) s[j] = pair_sum(v, j);
    float* part = a.part + (size_t)r.ph * kPartPhaseFloats;
    auto part_ptr = [&](int rg, int j, int row) {
        const int slot = rg == rf ? slot_rf : 0;
        return part + (((int64_t)(rg * 2 + slot) * kTilePairs + j) * kRows + row);
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
                if (!mbar_wait_warp(smem_u32(&sh.u_free[es][h][slot]), ph ^ 1u, abort, kEpiSleepNs)) return;
#pragma unroll
                for (int j = 0; j < kTilePairs; ++j) sh.u_box[es][h][slot][j][lane] = s[j];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.u_full[es][h][slot]));
                return;
            }
            if (!mbar_wait_warp(smem_u32(&sh.u_full[es][h][slot]), ph, abort, kEpiSleepNs)) return;
#pragma unroll
            for (int j = 0; j < kTilePairs; ++j) {
                g[j] = s[j];
                u[j] = sh.u_box[es][h][slot][j][lane];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.u_free[es][h][slot]));
        } else {
#pragma unroll
            for (int j = 0; j < kTilePairs; ++j)
                if (j < nrows) *part_ptr(blockIdx.x, j, m) = s[j];
            __syncwarp();   // the warp's stores come before lane 0's release
            if (lane == 0) old = atom_add_acq_rel(a.g_cnt + 2 * r.R + h, 1);
            if (__shfl_sync(0xffffffffu, old, 0) != 2 * nparts - 1) return;
            __syncwarp();   // the lanes' reads below come after lane 0's acquire
#pragma unroll
            for (int j = 0; j < kTilePairs; ++j) {
                g[j] = j < nrows ? part_total(part, rf, rl, slot_rf, j, 32 * h + lane) : 0.f;
                u[j] = j < nrows ? part_total(part, rf, rl, slot_rf, j, 64 + 32 * h + lane) : 0.f;
            }
        }
#pragma unroll 1
        for (int j = 0; j < nrows; ++j) {
            const float hv = __bfloat162float(__float2bfloat16_rn(silu_f(pick(g, j)) * pick(u, j)));
            store_h_digits(a, (int64_t)tile.q0 + j, 2 * rb + h, hv);
        }
        __syncwarp();
        if (lane == 0) red_release_add(a.h_flag + r.R, 1);
        return;
    }

    // down: this warp's 32 rows into the pairs' slots
    const int row = kRows * rb + m;
    if (nparts > 1) {
#pragma unroll
        for (int j = 0; j < kTilePairs; ++j)
            if (j < nrows) *part_ptr(blockIdx.x, j, m) = s[j];
        __syncwarp();
        if (lane == 0) old = atom_add_acq_rel(a.d_cnt + 4 * r.R + qd, 1);
        if (__shfl_sync(0xffffffffu, old, 0) != nparts - 1) return;
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kTilePairs; ++j) s[j] = j < nrows ? part_total(part, rf, rl, slot_rf, j, m) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < kTilePairs; ++j)
        if (j < nrows) a.stage[(int64_t)tile.pr[j] * a.H + row] = tile.w[j] * s[j];
    __syncwarp();   // the warp's stores come before lane 0's release
    if (lane == 0) old = atom_add_acq_rel(a.y_cnt + 4 * rb + qd, 1);
    if (__shfl_sync(0xffffffffu, old, 0) != n_tiles - 1) return;
    __syncwarp();
    // every tile's slots of these 32 rows are written: y = their sum per token
    // in j order (pairs left out never wrote a slot and add nothing)
    // (a token's ids and slots are loaded eight at a time, so their latencies
    // overlap; a slot left out may hold anything and is not added)
    for (int t = 0; t < a.T; ++t) {
        float acc = 0.f;
        for (int j0 = 0; j0 < a.k; j0 += 8) {
            int e[8];
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                e[u] = j < a.k ? __ldg(a.ids + t * a.k + j) : -1;
                x[u] = j < a.k ? __ldcg(a.stage + (int64_t)(t * a.k + j) * a.H + row) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) acc = (unsigned)e[u] < (unsigned)a.E ? acc + x[u] : acc;
        }
        __nv_bfloat16 yb = __float2bfloat16_rn(acc);
        a.y[(int64_t)t * a.H + row] = *reinterpret_cast<uint16_t*>(&yb);
    }
}

// Three barriers' phases complete (bounded as mbar_wait); the first polls are
// issued back to back so that their latencies overlap.
__device__ __forceinline__ bool mbar_wait3(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, uint32_t b3,
                                           uint32_t p3, volatile int* abort)
{
    const bool r1 = mbar_try_wait(b1, p1), r2 = mbar_try_wait(b2, p2), r3 = mbar_try_wait(b3, p3);
    if (r1 && r2 && r3) return true;
    return (r1 || mbar_wait_sleep(b1, p1, abort, kConsumerSleepNs)) &&
           (r2 || mbar_wait_sleep(b2, p2, abort, kConsumerSleepNs)) &&
           (r3 || mbar_wait_sleep(b3, p3, abort, kConsumerSleepNs));
}

// shared memory of a CTA: the static state and the rings at the largest scale rows
static_assert(sizeof(SharedState) + kOffS + 2 * kRows * kMaxScaleRow + 1024 <= 227 * 1024,
              "the CTA's shared memory fits an SM");

__global__ void __launch_bounds__(kThreads, 1)
decode_stream_kernel(const __grid_constant__ CUtensorMap gu_map, const __grid_constant__ CUtensorMap dn_map,
                     const __grid_constant__ CUtensorMap gu_sf_map, const __grid_constant__ CUtensorMap dn_sf_map,
                     const __grid_constant__ CUtensorMap xd_map, const __grid_constant__ CUtensorMap sxd_map,
                     const __grid_constant__ CUtensorMap hd_map, const __grid_constant__ CUtensorMap shd_map,
                     const __grid_constant__ StreamArgs a)
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
        for (int s = 0; s < kBSlotsMax; ++s) {
            mbar_init(smem_u32(&sh.full_b[s]), 1);
            mbar_init(smem_u32(&sh.empty_b[s]), kIssuers);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.a_full[s]), kCWarps / kGroups);
            mbar_init(smem_u32(&sh.a_empty[s]), 1);
        }
        for (int s = 0; s < kAccSets; ++s) {
            mbar_init(smem_u32(&sh.d_full[s]), kIssuers);
            mbar_init(smem_u32(&sh.d_empty[s]), kEWarps);
        }
        for (int e = 0; e < kESets; ++e)
            for (int h = 0; h < 2; ++h)
                for (int s = 0; s < 2; ++s) {
                    mbar_init(smem_u32(&sh.u_full[e][h][s]), 1);
                    mbar_init(smem_u32(&sh.u_free[e][h][s]), 1);
                }
        mbar_init(smem_u32(&sh.drain), kIssuers);
        sh.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh.tmem), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProdWarp && lane == 0) {
        prefetch_tmap(&gu_map);
        prefetch_tmap(&dn_map);
        prefetch_tmap(&gu_sf_map);
        prefetch_tmap(&dn_sf_map);
    }
    if (warp == kActWarp && lane == 0) {
        prefetch_tmap(&xd_map);
        prefetch_tmap(&sxd_map);
        prefetch_tmap(&hd_map);
        prefetch_tmap(&shd_map);
    }
    if (warp == 1) {
        // The step's tiles, from the routing itself (inputs: no need to wait for
        // the permutation kernel), in the order of their routed expert ids: each
        // kept expert gets ceil(pairs / 4) tiles and its pairs (ascending pair
        // index) are split evenly over them, as the permutation splits them.  A
        // tile's first row of h (q0) counts the kept pairs of smaller ids, so
        // the plain and the cached forward lay h out alike.  Behind an expert
        // cache the planes' index of expert r is its slot.  At most 32 pairs
        // (one per lane).
        int r = -1, plane = -1;
        // (every lane's router weight is loaded beside its id, so the two
        // loads' latencies overlap; the tiles pick them up from shared memory)
        sh.w_of[lane] = lane < a.P ? __ldg(a.weights + lane) : 0.f;
        if (lane < a.P) {
            r = __ldg(a.route_ids + lane);
            if (a.slot_of != nullptr) plane = (unsigned)r < (unsigned)a.n_route ? __ldg(a.slot_of + r) : -1;
            else plane = r;
            if ((unsigned)plane >= (unsigned)a.E) r = -1;
        }
        const int key = r >= 0 ? r : 0x7FFFFFFF;
        const uint32_t same = __match_any_sync(0xffffffffu, key);
        const bool lead = r >= 0 && (__ffs(same) - 1) == lane;
        const int cnt = __popc(same);
        const int ntl = lead ? (cnt + kTilePairs - 1) / kTilePairs : 0;
        int before = 0, total = 0, pbefore = 0;
        for (int u = 0; u < 32; ++u) {
            const int ku = __shfl_sync(0xffffffffu, key, u), nu = __shfl_sync(0xffffffffu, ntl, u);
            before += ku < key ? nu : 0;
            pbefore += ku < key ? 1 : 0;
            total += nu;
        }
        __syncwarp();
        for (int t = 0; t < ntl; ++t) {
            const int r0 = t * cnt / ntl, r1 = (t + 1) * cnt / ntl;
            TileInfo& ti = sh.tinfo[before + t];
            ti.q0 = pbefore + r0;
            ti.nrows = r1 - r0;
            uint32_t rest = same;   // the expert's pairs from its (r0 + j)-th on
            for (int j = 0; j < r0; ++j) rest &= rest - 1u;
            for (int j = 0; j < kTilePairs; ++j) {
                const int pr = j < r1 - r0 ? __ffs(rest) - 1 : 0;
                rest &= rest - 1u;
                ti.pr[j] = pr;
                ti.tok[j] = pr / a.k;
                ti.w[j] = j < r1 - r0 ? sh.w_of[pr] : 0.f;
            }
            sh.plane_of[before + t] = plane;
        }
        const int nm = __reduce_max_sync(0xffffffffu, lead ? (cnt + ntl - 1) / ntl : 0);
        if (lane == 0) {
            sh.n_tiles = total;
            sh.nmax = nm > 0 ? nm : 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh.tmem;
    volatile int* abort = &sh.abort_flag;
    const int n_tiles = sh.n_tiles;
    const int rbg = a.I / 64, rbd = a.H / 128;
    const int32_t Lg = a.H / kChunk, Ld = a.I / kChunk;
    if (tid == 0) {
        // this CTA's ranges of the four phases
        for (int p = 0; p < kPhases; ++p) {
            const bool gu = p < kTileGroups;
            const int gi = p % kTileGroups;   // tile group: tiles [gi n / G, (gi + 1) n / G) rounded up
            const int t0 = (gi * n_tiles + kTileGroups - 1) / kTileGroups;
            const int nt = ((gi + 1) * n_tiles + kTileGroups - 1) / kTileGroups - t0;
            const int rbn = gu ? rbg : rbd;
            const int32_t L = gu ? Lg : Ld;
            const Seq q(nt * rbn * L, L, (int32_t)gridDim.x);
            sh.pt.n[p] = q.n;
            sh.pt.t0[p] = t0;
            sh.pt.rbase[p] = t0 * rbn;
            sh.pt.start[p] = q.start(blockIdx.x);
            sh.pt.len[p] = q.start(blockIdx.x + 1) - sh.pt.start[p];
        }
    }
    __syncthreads();
    RunIter r0{};
    r0.pt = &sh.pt;
    r0.Lg = Lg;
    r0.Ld = Ld;
    const uint32_t sbuf0 = ring_addr + kOffS;
    const uint32_t sbytes = (uint32_t)kRows * (uint32_t)a.sb;   // one scale tile

    if (warp == kProdWarp) {
        // ------------------------------------------------ code and scale producers (read only inputs)
        if (lane == 0) {
            // every pair's code tile (128 rows x 128 code bytes: chunks c, c + 1)
            // in one tensor copy, into ring slot sp % kCSlots; first the scale
            // tile of run 0 (the scale lane, below, takes the runs after it), so
            // that it does not wait behind the ring's first code tiles
            {
                RunIter f = r0;
                if (f.next()) {
                    const bool gu = f.kind == 1;
                    const int rb = (int)(f.R % (gu ? rbg : rbd));
                    const int e = sh.plane_of[f.R / (gu ? rbg : rbd)];
                    const uint32_t fs = smem_u32(&sh.full_s[0]);
                    mbar_arrive_expect_tx_relaxed(fs, kRows * (uint32_t)(gu ? a.H / 32 : a.I / 32));
                    if (gu) tma_load_3d(sbuf0, &gu_sf_map, 0, 64 * rb, 2 * e, fs);
                    else tma_load_2d(sbuf0, &dn_sf_map, 0, e * a.H + kRows * rb, fs);
                }
            }
            RunIter it = r0;
            int sp = 0;
            bool stop = false;
            while (!stop && it.next()) {
                const bool gu = it.kind == 1;
                const int rb = (int)(it.R % (gu ? rbg : rbd));
                const int e = sh.plane_of[it.R / (gu ? rbg : rbd)];
                for (int jp = 0; jp < it.npairs; ++jp, ++sp) {
                    const uint32_t slot = (uint32_t)sp % kCSlots;
                    if (!mbar_wait_sleep(smem_u32(&sh.empty_c[slot]), (((uint32_t)sp / kCSlots) & 1u) ^ 1u, abort,
                                         kProducerSleepNs)) {
                        stop = true;
                        break;
                    }
                    const uint32_t base = ring_addr + slot * kCodeBytes, fb = smem_u32(&sh.full_c[slot]);
                    const int c = it.c0 + 2 * jp;
                    mbar_arrive_expect_tx_relaxed(fb, kCodeBytes);
                    // code bytes 64 c .. 64 c + 127 of every row
                    if (gu) {
                        // 64 gate rows then their 64 up rows (planes 2e, 2e + 1 of the
                        // w13 plane seen as 2E planes of I rows)
                        tma_load_3d(base, &gu_map, c * 64, 64 * rb, 2 * e, fb);
                    } else {
                        tma_load_2d(base, &dn_map, c * 64, e * a.H + kRows * rb, fb);
                    }
                }
            }
            if (*abort) {
                // the consumers may have stopped before the last tiles landed: wait
                // (bounded) for the copies of the last ring positions
                volatile int never = 0;
                for (int sq = sp > kCSlots ? sp - kCSlots : 0; sq < sp; ++sq)
                    (void)mbar_wait(smem_u32(&sh.full_c[sq % kCSlots]), ((uint32_t)sq / kCSlots) & 1u, &never);
            }
        } else if (lane == 1) {
            // every run's scale tile, in run order, into buffer g % 2 once run
            // g - 2 is done with it: a buffer's next tile is sent only after the
            // one before it was both sent and read, so no wait on the buffer can
            // mistake an older phase for the one it waits for
            RunIter it = r0;
            int last_g[2] = {-1, -1};   // the last run whose tile went to each buffer
            while (it.next()) {
                if (it.g == 0) {   // sent by the code lane
                    last_g[0] = 0;
                    continue;
                }
                const bool gu = it.kind == 1;
                const int rb = (int)(it.R % (gu ? rbg : rbd));
                const int e = sh.plane_of[it.R / (gu ? rbg : rbd)];
                const uint32_t b = (uint32_t)it.g & 1u;
                if (!mbar_wait_sleep(smem_u32(&sh.empty_s[b]), (((uint32_t)it.g >> 1) & 1u) ^ 1u, abort,
                                     kProducerSleepNs))
                    break;
                const uint32_t fs = smem_u32(&sh.full_s[b]);
                mbar_arrive_expect_tx_relaxed(fs, kRows * (uint32_t)(gu ? a.H / 32 : a.I / 32));
                if (gu) tma_load_3d(sbuf0 + b * sbytes, &gu_sf_map, 0, 64 * rb, 2 * e, fs);
                else tma_load_2d(sbuf0 + b * sbytes, &dn_sf_map, 0, e * a.H + kRows * rb, fs);
                last_g[b] = it.g;
            }
            if (*abort) {
                volatile int never = 0;
                for (int b = 0; b < 2; ++b)
                    if (last_g[b] >= 0)
                        (void)mbar_wait(smem_u32(&sh.full_s[b]), ((uint32_t)last_g[b] >> 1) & 1u, &never);
            }
        }
    } else {
        // Launched as a programmatic dependent of the permutation kernel: what
        // it writes (the x digits, zeroed counters) is read, by the activation
        // producer and the epilogues, only after this wait.
        if (warp == kActWarp || (warp >= kEpiWarp0 && warp < kEpiWarp0 + kESets * kEWarps))
            asm volatile("griddepcontrol.wait;" ::: "memory");
        if (warp == kActWarp) {
            // ------------------------------------------------ activation producer
            // (per pair of the tile, one digit-row box of both chunks and one
            // scale box)
            RunIter it = r0;
            BRing br(sh.nmax);
            int sp = 0;
            bool stop = false;
            int waited_ph = -1;   // the down phase whose h was last waited for
            while (!stop && it.next()) {
                if (it.kind == 0 && it.ph != waited_ph) {
                    // the down range of this phase reads h of every tile it touches:
                    // wait (bounded) until all of those 64-element blocks are published
                    waited_ph = it.ph;
                    const int32_t ds = sh.pt.start[it.ph], dn = sh.pt.len[it.ph];
                    const int t0 = sh.pt.t0[it.ph] + ds / Ld / rbd, t1 = sh.pt.t0[it.ph] + (ds + dn - 1) / Ld / rbd;
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
                const TileInfo& tile = sh.tinfo[it.R / (it.kind == 1 ? rbg : rbd)];
                for (int jp = 0; jp < it.npairs; ++jp, ++sp, br.advance()) {
                    const uint32_t slot = br.slot;
                    int ok = 1;
                    if (lane == 0)
                        ok = mbar_wait_sleep(smem_u32(&sh.empty_b[slot]), br.phase ^ 1u, abort, kProducerSleepNs);
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        stop = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&sh.full_b[slot]);
                    if (lane == 0)
                        mbar_arrive_expect_tx_relaxed(fb, (uint32_t)tile.nrows * (kActDigits * (2 * 128 + 16)));
                    __syncwarp();
                    if (lane < tile.nrows) {
                        // pair `lane` of the tile: gate_up reads its token's rows of x, down its rows of h
                        const int brow = kActDigits * (it.kind == 1 ? tile.tok[lane] : tile.q0 + lane);
                        const int c = it.c0 + 2 * jp;
                        const uint32_t base = ring_addr + kOffB + slot * br.stride;
                        // {128 bytes, 8 rows, chunks c and c + 1}: chunk-major, pair lane's tiles
                        tma_load_3d(base + (2 * lane) * kBTile, it.kind == 1 ? &xd_map : &hd_map, 0, brow, c,
                                    fb);
                        tma_load_2d(base + br.sfoff + lane * (kActDigits * 16), it.kind == 1 ? &sxd_map : &shd_map,
                                    c * 8, brow, fb);
                    }
                }
            }
            if (*abort && lane == 0) {
                volatile int never = 0;
                const int nb = (int)br.nb;
                for (int sq = sp > nb ? sp - nb : 0; sq < sp; ++sq)
                    (void)mbar_wait(smem_u32(&sh.full_b[sq % nb]), ((uint32_t)sq / (uint32_t)nb) & 1u, &never);
            }
        } else if (warp >= kMmaWarp0) {
            // ------------------------------------------------ MMA issuers
            // Issuer q takes chunk q of every pair (its own accumulator of the run's
            // set, its group's A stages); each also commits the B slot it read,
            // which is free once both chunks of the pair are done.  (Issuers in
            // separate warps: one warp issues its tcgen05.mma instructions one
            // after the other.)
            const int q = warp - kMmaWarp0;
            if (lane == 0) {
                RunIter it = r0;
                BRing br(sh.nmax);
                int sp = 0;
                bool stop = false;
                while (!stop && it.next()) {
                    const uint32_t set = (uint32_t)it.g % kAccSets;
                    // The accumulator set of run g is free once the epilogue of run
                    // g - kAccSets read it.  Both issuers wait at every run's start:
                    // d_full[set] takes one commit from each, so neither may commit
                    // for a later run of the set before the epilogue of this one
                    // has seen both of its commits.
                    if (it.g >= kAccSets &&
                        !mbar_wait_sleep(smem_u32(&sh.d_empty[set]), (((uint32_t)it.g / kAccSets) - 1u) & 1u, abort,
                                         kIssuerSleepNs))
                        break;
                    const uint32_t d = tm + 32u * (2u * set + (uint32_t)q);
                    for (int jp = 0; jp < it.npairs; ++jp, ++sp, br.advance()) {
                        const uint32_t st = (uint32_t)(kGStages * q) + (uint32_t)sp % kGStages, bs = br.slot;
                        const bool ready = mbar_wait_sleep(smem_u32(&sh.full_b[bs]), br.phase, abort,
                                                           kIssuerSleepNs) &&
                                           mbar_wait_sleep(smem_u32(&sh.a_full[st]), ((uint32_t)sp / kGStages) & 1u,
                                                           abort, kIssuerSleepNs);
                        if (!ready) {
                            stop = true;
                            break;
                        }
                        tc_fence_after();
                        // this chunk's B tiles: pair j at (2 j + q) kBTile of the slot
                        const uint64_t bd = smem_desc_sw128_sbo(
                            ring_addr + kOffB + bs * br.stride + (uint32_t)q * kBTile, 2 * kBTile);
                        // MMA t: K 64t..64t+63 of the chunk = A columns 8t..8t+7 of the
                        // stage, 32 bytes of every B row, scale word t / 2, bytes
                        // 2 (t % 2) and 2 (t % 2) + 1
#pragma unroll
                        for (uint32_t t = 0; t < 4; ++t)
                            umma_mxf4_ts(d, tm + kColA + 32 * st + 8 * t, bd + 2 * t,
                                         idesc_mxf4(kRows, kN, 2 * (t & 1), 2 * (t & 1)),
                                         tm + kColSfa + 8 * st + 4 * (t >> 1), tm + kColSfb + 8 * st + 4 * (t >> 1),
                                         (jp > 0 || t != 0) ? 1u : 0u);
                        umma_commit(smem_u32(&sh.a_empty[st]));
                        umma_commit(smem_u32(&sh.empty_b[bs]));
                    }
                    if (!stop) umma_commit(smem_u32(&sh.d_full[set]));
                }
                // every MMA of both issuers has completed before tensor memory is freed
                umma_commit(smem_u32(&sh.drain));
                volatile int never = 0;
                (void)mbar_wait(smem_u32(&sh.drain), 0u, &never);
            }
        } else if (warp >= kEpiWarp0) {
            // ------------------------------------------------ epilogue warps
            // set e takes the runs g with g % kESets == e, so one run's epilogue
            // overlaps the next one's
            const uint32_t tq = tm + ((uint32_t)(32 * (warp & 3)) << 16);
            const int es = (warp - kEpiWarp0) / kEWarps;
            RunIter it = r0;
            int wn = 0;
            while (it.next()) {
                if (it.g % kESets != es) continue;
                epilogue(a, sh, tq, Run{it.kind, it.R, it.g, it.ph, it.Rl}, n_tiles, wn, abort);
                // whole gate_up row blocks use the u_box slots in turn
                if (it.kind == 1) {
                    const Seq q(sh.pt.n[it.ph], Lg, (int32_t)gridDim.x);
                    if (q.range_of(it.Rl * Lg) == q.range_of((it.Rl + 1) * Lg - 1)) ++wn;
                }
            }
        } else {
            // ------------------------------------------------ consumers
            const int h = warp / (kCWarps / kGroups), qd = warp & 3;   // group, lane quadrant
            const int m = 32 * qd + lane;                               // weight row of the row block
            const uint32_t tq = tm + ((uint32_t)(32 * qd) << 16);
            const uint32_t swz = (uint32_t)m & 7u;   // 128B swizzle of this code row
            uint32_t bad_scale = 0;
            RunIter it = r0;
            BRing br(sh.nmax);
            int sp = 0;
            bool stop = false;
            while (!stop && it.next()) {
                const uint32_t sbuf = (uint32_t)it.g & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.full_s[sbuf]), ((uint32_t)it.g >> 1) & 1u, abort)))
                    break;
                // the row's scale words of chunk c0 + h (8 bytes per chunk)
                const uint32_t srow = sbuf0 + sbuf * sbytes +
                                      (uint32_t)m * (uint32_t)(it.kind == 1 ? a.H / 32 : a.I / 32) +
                                      8u * (uint32_t)(it.c0 + h);
                for (int jp = 0; jp < it.npairs; ++jp, ++sp, br.advance()) {
                    const uint32_t cs = (uint32_t)sp % kCSlots, bs = br.slot;
                    const uint32_t st = (uint32_t)(kGStages * h) + (uint32_t)sp % kGStages;
                    // the code tile and the stage first: the expansion does not need
                    // the activation rows, whose scale words are stored last
                    const bool got = mbar_wait2(smem_u32(&sh.full_c[cs]), ((uint32_t)sp / kCSlots) & 1u,
                                                smem_u32(&sh.a_empty[st]), (((uint32_t)sp / kGStages) & 1u) ^ 1u, abort);
                    if (!__all_sync(0xffffffffu, got)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    // the row's 64 code bytes of chunk h of the pair (16-byte unit
                    // 4 h + u of the 128-byte row at (4 h + u) ^ swz), its two scale
                    // words, and the digit rows' scale words (B row n = lane: its
                    // 16-byte group of the pair at sfoff + 16 n, word h; rows of
                    // pairs past the tile's read whatever lies there, and only
                    // their own, unused, accumulator columns see it)
                    const uint32_t cb = ring_addr + cs * kCodeBytes + (uint32_t)m * 128u;
                    uint32_t wd[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 v = lds_u4(cb + (((4u * (uint32_t)h + (uint32_t)u) ^ swz) << 4));
                        wd[4 * u] = v.x;
                        wd[4 * u + 1] = v.y;
                        wd[4 * u + 2] = v.z;
                        wd[4 * u + 3] = v.w;
                    }
                    uint2 sfa = lds_u2(srow + 16u * (uint32_t)jp);
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&sh.empty_c[cs]));
                        if (jp == it.npairs - 1) mbar_arrive(smem_u32(&sh.empty_s[sbuf]));
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
                    tmem_st_a_sfa(tq + kColA + 32 * st, r, tq + kColSfa + 8 * st + (uint32_t)qd, sfa.x,
                                  tq + kColSfa + 8 * st + 4 + (uint32_t)qd, sfa.y);
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.full_b[bs]), br.phase, abort))) {
                        tmem_st_sfb_wait(r, sfa.x, sfa.y, tq + kColSfb + 8 * st, 0u, tq + kColSfb + 8 * st + 4, 0u);
                        stop = true;
                        break;
                    }
                    const uint2 sfb =
                        lds_u2(ring_addr + kOffB + bs * br.stride + br.sfoff + (uint32_t)lane * 16u + 8u * (uint32_t)h);
                    tmem_st_sfb_wait(r, sfa.x, sfa.y, tq + kColSfb + 8 * st, sfb.x, tq + kColSfb + 8 * st + 4, sfb.y);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.a_full[st]));
                }
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

size_t stream_part_floats() { return (size_t)kPhases * kPartPhaseFloats; }

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
    a.weights = weights;
    a.ids = ids;
    a.route_ids = route_ids;
    a.slot_of = slot_of;
    a.n_route = n_route;
    a.hd = ws.hd;
    a.shd = ws.shd;
    a.stage = ws.stage;
    a.part = ws.gu_part;
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
    // activation digit rows ([rows][K/2] bytes) seen as {128 bytes of a chunk,
    // row, chunk}, the chunk stride (128) below the row stride: a box of one
    // pair's 8 rows x 2 chunks lands chunk-major, each chunk's 8 rows one
    // 128B-swizzle atom of the UMMA B operand; and their 16-byte scale groups
    // (two chunks)
    CUtensorMap xd_map, sxd_map, hd_map, shd_map;
    const int64_t xdims[3] = {128, (int64_t)kActDigits * T, H / kChunk}, xstr[2] = {H / 2, 128};
    const int64_t hdims[3] = {128, (int64_t)kActDigits * P, I / kChunk}, hstr[2] = {I / 2, 128};
    const uint32_t dbox[3] = {128, (uint32_t)kActDigits, 2};
    if ((e = make_tmap_u8(&xd_map, ws.xd, 3, xdims, xstr, dbox, 128)) != cudaSuccess ||
        (e = make_tmap_2d(&sxd_map, ws.sxd, false, (int64_t)kActDigits * T, H / 32, 16, kActDigits, 0)) != cudaSuccess ||
        (e = make_tmap_u8(&hd_map, ws.hd, 3, hdims, hstr, dbox, 128)) != cudaSuccess ||
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
