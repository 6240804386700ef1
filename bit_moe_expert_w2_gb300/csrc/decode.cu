// Decode path (T <= 64): the 2-bit planes of every active expert are streamed
// from HBM once per layer and multiplied on the tensor cores in block-scaled FP4
// (tcgen05.mma kind::mxf4).
//
// vLLM-Moet, page "vLLM-Moet wiki", section "The kernels": codes expanded in
// registers and fed to block-scaled tensor-core MMAs; section "FP4 recovery":
// decode is HBM-bound, the 2-bit read is the cost.  Page "The v0.24.0 port",
// section "Benchmarks": tokens grouped by expert, so each active expert's
// weights are read once per step however many tokens use it.  Page "The
// v0.24.0 port", "Deterministic unpermute" bullet: per-pair results are placed
// in their own slot and summed in a fixed order.
//
// Why block-scaled fp4 operands (tcgen05.mma kind::mxf4, scale_vec::2X): a
// weight is +-1 or +-4 times 2^(s-127) with one UE8M0 byte s per 32 K of a row,
// which is an e2m1 value under an MX block scale.  The tensor core applies s
// itself, so the expansion is one nibble per code, (c << 2) | 2: per 16-code
// word one shift and two and-or operations, with no table.  Activations enter
// as kActDigits rows of e2m1 digits each (fp4_elem order, digit_scale_byte).
// Packed operands need one MMA of K = 64 per 64 codes of a row, so a 256-K
// chunk of a row is 32 TMEM columns.
//
// Work items (one global queue, every gate_up unit before any down item; each
// CTA's first item is its own block index, the rest come from an atomic
// counter):
//   gate_up  (tile of <= 4 pairs of one expert, 64-row block): the block's 64
//            gate rows and its 64 up rows over the whole K = H.  Its epilogue
//            writes h = bf16(SiLU(g) * u) of those 64 elements as digit rows and
//            publishes them with one release add per 32 elements.  When the
//            units are at most half the CTAs (the smallest steps), each is two
//            items over the two halves of K: both store fp32 partial sums, and
//            the last of the unit's eight consumer warps to arrive adds the two
//            (an order-free sum of two terms) and writes h.
//   down     (tile, 128-row block of W_down, K segment of I): its epilogue
//            writes w * (W_down h) into the pair's fp32 slot of that segment; a
//            dependent combine kernel sums every token's slots in (j, segment)
//            order into y.

// Each CTA has six warps:
//   warp 4     producer: takes items from the queue, publishes them, and streams
//              every 256-K chunk into two rings of shared-memory slots: the code
//              tile (128 rows x 64 bytes, 64B-swizzled) and the 16-byte scale
//              group of every weight row by TMA into a code slot (barrier
//              full_a), freed by the consumer warps as soon as they hold the
//              chunk in registers; the eight activation digit rows of each pair
//              of the tile (one TMA box of 8 rows x 128 bytes, landing in the
//              128B-swizzled UMMA layout) with their scale groups by TMA into an
//              activation slot (full_b), freed by the MMA that reads it.  A down item's code chunks go out at once; its
//              activation rows (h) only after the gate_up units that write them
//              have published them.
//   warps 0-3  consumers, one per TMEM lane quadrant and one thread per weight
//              row: expand the row's 256 codes of a chunk to packed e2m1, store
//              them with the row's two scale words and this quadrant's copy of
//              the digit rows' scale words into TMEM; then the item epilogues
//   warp 5     MMA issuer (one thread): 4 x tcgen05.mma (M=128, N=32, K=64) per
//              chunk into the TMEM accumulator
// An item's accumulator is read by the consumer warps after they stored the
// first chunk of the next item, or before the next item when that is a down item
// (whose data may wait for h: no epilogue is held across that wait); the next
// item's first MMA waits until it has been read.  (An MMA costs its issuing
// thread the same whatever N is, so a tile takes four pairs of eight digit rows,
// N = 32, in one accumulator rather than two pairs in each of two.)
// Every wait is bounded; on a timeout the kernel raises the pipeline status bit,
// drains its MMAs, frees its tensor memory and returns.
#include <algorithm>

#include "tc.cuh"

namespace moe_w2 {

namespace {

constexpr int kChunk = 256;                          // K per chunk: 4 MMAs of K = 64 (two scale blocks each)
constexpr int kRows = 128;                           // weight rows per item (MMA M)
constexpr int kTilePairs = 4;                        // pairs per tile
constexpr int kN = 32;                               // MMA N: the digit rows of the tile's pairs
static_assert(kActDigits * kTilePairs <= kN, "a tile's digit rows must fit the MMA N");
constexpr int kCWarps = 4;                           // consumer warps
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kCSlots = 3;                           // code slots (freed once the consumers hold the chunk)
constexpr int kBSlots = 4;                           // activation slots (freed by the MMA that reads them)
constexpr uint32_t kCodeBytes = kRows * 64;          // 128 rows x 64 code bytes, 64B-swizzled
constexpr uint32_t kBBytes = kN * 128;               // 32 digit rows x 128 bytes (256 e2m1), 128B-swizzled
constexpr uint32_t kSfaBytes = kRows * 16;           // 16-byte scale groups (2 chunks) of the 128 weight rows
constexpr uint32_t kSfbBytes = kN * 16;              // the same for the 16 digit rows
constexpr uint32_t kOffB = kCSlots * kCodeBytes;     // ring: code tiles, activation tiles (1024-aligned),
constexpr uint32_t kOffSfa = kOffB + kBSlots * kBBytes;      // then the scale groups
constexpr uint32_t kOffSfb = kOffSfa + kCSlots * kSfaBytes;
constexpr uint32_t kRingBytes = kOffSfb + kBSlots * kSfbBytes;
constexpr int kInfo = 8;                             // published items in flight
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kColD = 0;                        // accumulator: 32 columns
constexpr uint32_t kColA = 32;                       // A stages: 2 x 32 columns (256 K of e2m1)
constexpr uint32_t kColSfa = 96;                     // stage s, word w, quadrant q: column 96 + 8s + 4w + q
constexpr uint32_t kColSfb = 112;                    // stage s, word w: column 112 + 8s + 4w
// (scale-factor operands start on a 4-column boundary: an M = 128 tile's A
// scales span 4 columns, one per lane quadrant; a chunk has two scale words)
constexpr int32_t kHPublished = 2;                   // release adds per 64-element block of h (one per 32)

struct LayerArgs {
    int32_t H, I, T, k, E;
    DecodeSplit split;
    int64_t P;
    const int4* tiles;
    const int32_t* tile_count;
    const int32_t* sorted;
    const float* weights;
    const uint8_t* xd;           // [8T][H/2] digit rows of x
    const uint8_t* sxd;          // [8T][H/32]
    uint8_t* hd;                 // [8P][I/2] digit rows of h
    uint8_t* shd;                // [8P][I/32]
    float* stage;                // [s_dn][P][H]
    float* gu_part;              // [2][P][2I] gate_up partial sums of the K halves (null: no split)
    int32_t* h_flag;             // [tiles][I/64]: release adds once h of the block is written
    int32_t* gu_cnt;             // [tiles][I/64]: consumer warps of both K halves done with their partials
    int32_t* queue;
    const int32_t* ids;          // [T][k]
    DepWait dep;                 // the h wait: target bias and limit
    uint32_t* status;
};

struct SharedState {
    uint64_t full_a[kCSlots];    // producer -> consumers: code tile and weight-row scale groups landed (tx bytes)
    uint64_t empty_a[kCSlots];   // consumer warps -> producer: code slot read
    uint64_t full_b[kBSlots];    // producer -> consumers, MMA: digit rows and their scale groups landed (32 cp.async)
    uint64_t empty_b[kBSlots];   // MMA commit -> producer: activation slot read
    uint64_t a_full[2];          // consumer warps -> MMA: A stage written
    uint64_t a_empty[2];         // MMA commit -> consumers: A stage read
    uint64_t d_full;             // MMA commit -> consumers: accumulator complete
    uint64_t d_empty;            // consumer warps -> MMA: accumulator read
    uint64_t u_ready[2];         // up-row warps -> gate-row warps: up sums in u_buf
    uint64_t info_full[kInfo];   // producer -> consumers, MMA: item published
    uint64_t info_empty[kInfo];  // consumers, MMA -> producer: item done with
    uint64_t drain;
    int info[kInfo][12];         // published items (Item fields; kind -1 at the end)
    float u_buf[2][kTilePairs][64];
    uint32_t tmem;
    int abort_flag;
};

// A work item: one tile, 128 weight rows (gate_up: a 64-row block of gate and
// of up; down: a 128-row block of W_down) and the K chunks [c0, c1).
// seg: the down K segment, or the gate_up K half; nsplit: 2 for a gate_up unit
// split into two K halves, else 1.
struct Item {
    int kind;   // 1 gate_up, 0 down, -1 end
    int ti, rb, seg, c0, c1, expert, q0, nrows, nsplit;
};

__device__ __forceinline__ void put_item(int* dst, const Item& m)
{
    dst[0] = m.kind; dst[1] = m.ti; dst[2] = m.rb; dst[3] = m.seg; dst[4] = m.c0;
    dst[5] = m.c1; dst[6] = m.expert; dst[7] = m.q0; dst[8] = m.nrows; dst[9] = m.nsplit;
}
__device__ __forceinline__ Item get_item(const int* src)
{
    Item m;
    m.kind = src[0]; m.ti = src[1]; m.rb = src[2]; m.seg = src[3]; m.c0 = src[4];
    m.c1 = src[5]; m.expert = src[6]; m.q0 = src[7]; m.nrows = src[8]; m.nsplit = src[9];
    return m;
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t* p)
{
    int32_t v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Add with release semantics at GPU scope: this thread's earlier writes, and
// those it has observed (the warp's, after __syncwarp), are visible to a thread
// that reads the new value with ld_acquire.
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

// Position in a ring of N slots: slot q % N and phase bit (q / N) & 1 of the
// running chunk count q, stepped without a division.
template <uint32_t N>
struct RingPos {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void step()
    {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

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
__device__ __forceinline__ void store_h_digits(const LayerArgs& a, int64_t q, int blk, float v)
{
    const int lane = threadIdx.x & 31;
    const int pos = (lane & 16) | fp4_pos(lane & 15);
#pragma unroll
    for (int d = 0; d < kActDigits; ++d) {
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
        const uint32_t sd = digit_scale_byte(__uint_as_float(amax_bits));
        float qv;
        const uint32_t nib = e2m1_digit_hw(v * digit_inv_scale(sd), qv);
        v -= qv * digit_scale(sd);
        const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 2);
        const int64_t row = kActDigits * q + d;
        if ((pos & 1) == 0) a.hd[row * (a.I / 2) + blk * 16 + (pos >> 1)] = (uint8_t)(nib | (other << 4));
        if (lane == 0) a.shd[row * (a.I / 32) + blk] = (uint8_t)sd;
    }
}

// Epilogue of an item on the consumer warps: item n of this CTA (accumulator
// phase n & 1), and for gate_up its gn-th gate_up epilogue (u_buf and u_ready
// gn & 1).
//   gate_up  warps 2-3 (the up rows) hand their sums to warps 0-1 through
//            shared memory; warps 0-1 (the gate rows) form h = bf16(SiLU(g) * u)
//            for 32 elements each, write its digit rows and publish them
//   down     every warp writes w * (its rows of W_down h) into the pairs' slots
// u_buf[gn & 1] is written again only for gate_up epilogue gn + 2, which the
// up-row warps reach after the MMA took an A stage from the gate-row warps that
// those wrote after they finished epilogue gn.
__device__ __noinline__ void epilogue(const LayerArgs& a, SharedState& sh, uint32_t tq, const Item& it, int n,
                                      int gn, volatile int* abort)
{
    const int lane = threadIdx.x & 31, m = threadIdx.x, warp = m >> 5;
    const uint32_t ph = (uint32_t)n & 1u;
    const uint32_t ub = (uint32_t)gn & 1u, uph = ((uint32_t)gn >> 1) & 1u;
    // every lane waits (each acquires); the outcome is made warp-uniform before
    // the .sync.aligned tensor-memory load
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.d_full), ph, abort))) return;
    tc_fence_after();
    float v[32];
    tmem_ld32(tq + kColD, v);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sh.d_empty));
    if (it.kind == 1 && it.nsplit == 2) {
        // K half it.seg: the partial sums of this warp's 32 rows, then count the
        // warp in; the unit's last warp (of 2 x 4) adds both halves and writes h
        const int I2 = 2 * a.I;
        const int col = m < 64 ? 64 * it.rb + m : a.I + 64 * it.rb + (m - 64);
#pragma unroll
        for (int j = 0; j < kTilePairs; ++j)
            if (j < it.nrows) a.gu_part[((int64_t)it.seg * a.P + it.q0 + j) * I2 + col] = pair_sum(v, j);
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel(a.gu_cnt + it.ti * (a.I / 64) + it.rb, 1) == 2 * kCWarps - 1;
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __syncwarp();   // the lanes' loads below come after lane 0's acquire
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            const int i = 64 * it.rb + 32 * blk + lane;   // element of h
            for (int j = 0; j < it.nrows; ++j) {
                const float* p0 = a.gu_part + ((int64_t)it.q0 + j) * I2;
                const float* p1 = p0 + a.P * I2;
                const float g = __ldcg(p0 + i) + __ldcg(p1 + i);
                const float u = __ldcg(p0 + a.I + i) + __ldcg(p1 + a.I + i);
                const float hv = __bfloat162float(__float2bfloat16_rn(silu_f(g) * u));
                store_h_digits(a, (int64_t)it.q0 + j, 2 * it.rb + blk, hv);
            }
        }
        __syncwarp();
        if (lane == 0) red_release_add(a.h_flag + it.ti * (a.I / 64) + it.rb, kHPublished);
    } else if (it.kind == 1) {
        if (warp >= 2) {
#pragma unroll
            for (int j = 0; j < kTilePairs; ++j) sh.u_buf[ub][j][m - 64] = pair_sum(v, j);
            mbar_arrive(smem_u32(&sh.u_ready[ub]));   // every lane: its own stores are released
            return;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.u_ready[ub]), uph, abort))) return;
        const int blk = 2 * it.rb + warp;   // the 32 elements 64 rb + 32 warp + lane of h
#pragma unroll
        for (int j = 0; j < kTilePairs; ++j)
            if (j < it.nrows) {
                const float g = pair_sum(v, j), u = sh.u_buf[ub][j][m];
                const float hv = __bfloat162float(__float2bfloat16_rn(silu_f(g) * u));
                store_h_digits(a, (int64_t)it.q0 + j, blk, hv);
            }
        __syncwarp();
        if (lane == 0) red_release_add(a.h_flag + it.ti * (a.I / 64) + it.rb, 1);
    } else {
        const int row = 128 * it.rb + m;
#pragma unroll
        for (int j = 0; j < kTilePairs; ++j)
            if (j < it.nrows) {
                const int pr = __ldg(a.sorted + it.q0 + j);
                a.stage[((int64_t)it.seg * a.P + pr) * a.H + row] = __ldg(a.weights + pr) * pair_sum(v, j);
            }
    }
}

__global__ void __launch_bounds__(kThreads, 4)
decode_layer_kernel(const __grid_constant__ CUtensorMap gu_map, const __grid_constant__ CUtensorMap dn_map,
                    const __grid_constant__ CUtensorMap gu_sf_map, const __grid_constant__ CUtensorMap dn_sf_map,
                    const __grid_constant__ CUtensorMap xd_map, const __grid_constant__ CUtensorMap sxd_map,
                    const __grid_constant__ CUtensorMap hd_map, const __grid_constant__ CUtensorMap shd_map,
                    const LayerArgs a)
{
    __shared__ SharedState sh;
    extern __shared__ uint8_t dyn_smem[];   // kRingBytes + 1024 (aligned below)
    const uint32_t ring_addr = (smem_u32(dyn_smem) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kCSlots; ++s) {
            mbar_init(smem_u32(&sh.full_a[s]), 1);
            mbar_init(smem_u32(&sh.empty_a[s]), kCWarps);
        }
        for (int s = 0; s < kBSlots; ++s) {
            mbar_init(smem_u32(&sh.full_b[s]), 1);
            mbar_init(smem_u32(&sh.empty_b[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sh.a_full[s]), kCWarps);
            mbar_init(smem_u32(&sh.a_empty[s]), 1);

            mbar_init(smem_u32(&sh.u_ready[s]), 64);
        }
        for (int s = 0; s < kInfo; ++s) {
            mbar_init(smem_u32(&sh.info_full[s]), 1);
            mbar_init(smem_u32(&sh.info_empty[s]), kCWarps + 1);
        }
        mbar_init(smem_u32(&sh.d_full), 1);
        mbar_init(smem_u32(&sh.d_empty), kCWarps);
        mbar_init(smem_u32(&sh.drain), 1);
        sh.abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&sh.tmem), kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tmap(&gu_map);
        prefetch_tmap(&dn_map);
        prefetch_tmap(&gu_sf_map);
        prefetch_tmap(&dn_sf_map);
        prefetch_tmap(&xd_map);
        prefetch_tmap(&sxd_map);
        prefetch_tmap(&hd_map);
        prefetch_tmap(&shd_map);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = sh.tmem;
    volatile int* abort = &sh.abort_flag;

    // Launched as a programmatic dependent of the permutation kernel: the setup
    // above overlaps it; everything it writes (tiles, counters, x digits) is read
    // only after this wait.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next kernel on the stream may be scheduled now (a dependent launch
    // waits for this grid to finish before it reads its results)
    asm volatile("griddepcontrol.launch_dependents;");
    const int n_tiles = *a.tile_count;
    const int rbg = a.I / 64, rbd = a.H / 128;
    const int nch_gu = a.H / kChunk, nch_dn = a.I / kChunk;
    // gate_up units split into two K halves when they are at most half the CTAs
    const int nsplit = (a.gu_part != nullptr && 2 * (int64_t)n_tiles * rbg <= (int64_t)gridDim.x) ? 2 : 1;
    const int64_t n_gu = (int64_t)n_tiles * rbg * nsplit;
    const int64_t n_dn = (int64_t)n_tiles * rbd * a.split.s_dn;

    if (warp == kProducerWarp) {
        // ------------------------------------------------ producer
        RingPos<kCSlots> cp;   // code ring
        RingPos<kBSlots> bp;   // activation ring
        uint32_t issued = 0;   // code tiles issued (code ring positions 0 .. issued-1)
        uint32_t issued_b = 0; // activation tiles issued
        int ahead = 0;         // the queue index taken one item ahead (lane 0)
        int n = 0;
        bool ok = true;
        // publish one item; false when the pipeline gave up
        auto publish = [&](const Item& m) {
            const uint32_t islot = (uint32_t)n % kInfo;
            int w = 1;
            if (lane == 0) w = mbar_wait(smem_u32(&sh.info_empty[islot]), (((uint32_t)n / kInfo) & 1u) ^ 1u, abort);
            if (!__shfl_sync(0xffffffffu, w, 0)) return false;
            if (lane == 0) {
                put_item(sh.info[islot], m);
                mbar_arrive(smem_u32(&sh.info_full[islot]));
            }
            ++n;
            return true;
        };
        // wait (bounded) for a free slot at ring position p of a ring with barriers `empty`
        auto slot_free = [&](const uint64_t* empty, uint32_t slot, uint32_t phase) {
            int w = 1;
            if (lane == 0) w = mbar_wait(smem_u32(&empty[slot]), phase ^ 1u, abort);
            return __shfl_sync(0xffffffffu, w, 0) != 0;
        };
        // the code tile and the weight rows' scale groups of chunk ch (lane 0)
        auto load_codes = [&](const Item& m, int ch, uint32_t slot) {
            const uint32_t base = ring_addr + slot * kCodeBytes, fb = smem_u32(&sh.full_a[slot]);
            const uint32_t sfbase = ring_addr + kOffSfa + slot * kSfaBytes;
            // the 16-byte group of scale bytes (2 chunks) holding this chunk's two
            // words, for every weight row; every slot gets its own copy, so a
            // consumer reads words 2 (ch % 2) and 2 (ch % 2) + 1 of its own slot
            const int gx = (ch & ~1) * 8;
            mbar_arrive_expect_tx_relaxed(fb, kCodeBytes + kRows * 16);
            if (m.kind == 1) {
                // one box holds the row block's 64 gate rows, then its 64 up rows
                // (planes 2e and 2e + 1 of the w13 plane seen as 2E planes of I rows)
                tma_load_3d(base, &gu_map, ch * 64, 64 * m.rb, 2 * m.expert, fb);
                tma_load_3d(sfbase, &gu_sf_map, gx, 64 * m.rb, 2 * m.expert, fb);
            } else {
                const int rd = m.expert * a.H + 128 * m.rb;
                tma_load_2d(base, &dn_map, ch * 64, rd, fb);
                tma_load_2d(sfbase, &dn_sf_map, gx, rd, fb);
            }
        };
        // the h blocks a down item reads (64 elements each; four per chunk) are
        // published (bounded wait): lane r watches blocks 4 c0 + r, 4 c0 + r + 32, ...
        auto h_ready = [&](const Item& m) {
            const int32_t* hs = a.h_flag + m.ti * rbg;
            const int hb0 = (kChunk / 64) * m.c0, hb1 = (kChunk / 64) * m.c1;
            auto all_ready = [&]() {
                bool r = true;
                for (int hb = hb0 + lane; hb < hb1; hb += 32) r = r && ld_acquire(hs + hb) >= kHPublished + a.dep.bias;
                return __all_sync(0xffffffffu, r);
            };
            if (!all_ready()) {
                const long long t0 = clock64();
                bool timed_out = false;
                while (!all_ready()) {
                    if (__shfl_sync(0xffffffffu, *abort, 0)) break;
                    if (clock64() - t0 > a.dep.limit) {
                        timed_out = true;
                        break;
                    }
                    __nanosleep(64);
                }
                if (timed_out && lane == 0) *abort = 1;
            }
            __syncwarp();   // every lane's copies come after the lanes' acquires
            return __shfl_sync(0xffffffffu, *abort, 0) == 0;
        };
        // stream the chunks of a published item into the ring
        // publish an item and stream its chunks into the rings; `ahead` is taken
        // from the queue once the item is published
        auto stream = [&](const Item& m, bool first) {
            const bool gu = m.kind == 1;
            // the first chunks' code tiles go out before the activation rows: for a
            // down item, before the wait for h; for the CTA's first item, while
            // the ring is empty, before the loads that locate the rows
            const int npre = (!gu || first) ? min(m.c1 - m.c0, kCSlots) : 0;
            int ch = m.c0;
            for (int i = 0; i < npre; ++i, ++ch, cp.step()) {
                if (!slot_free(sh.empty_a, cp.slot, cp.phase)) return false;
                if (lane == 0) load_codes(m, ch, cp.slot);
            }
            issued += (uint32_t)npre;
            if (!publish(m)) return false;
            if (lane == 0) ahead = atomicAdd(a.queue, 1);
            // digit-row coordinate of the tile's pair `lane` (lanes < nrows):
            // gate_up the token's rows of x, down the pair's rows of h
            const int brow = lane < m.nrows
                                 ? kActDigits * (gu ? __ldg(a.sorted + m.q0 + lane) / a.k : m.q0 + lane)
                                 : 0;
            const CUtensorMap* bmap = gu ? &xd_map : &hd_map;
            const CUtensorMap* sbmap = gu ? &sxd_map : &shd_map;
            // the digit rows and their scale groups of chunk c into the next
            // activation slot: lane j < nrows copies pair j's 8 rows
            auto load_b = [&](int c) {
                if (!slot_free(sh.empty_b, bp.slot, bp.phase)) return false;
                const uint32_t fb = smem_u32(&sh.full_b[bp.slot]);
                if (lane == 0) mbar_arrive_expect_tx_relaxed(fb, (uint32_t)m.nrows * (kActDigits * (128 + 16)));
                __syncwarp();
                if (lane < m.nrows) {
                    const uint32_t base = ring_addr + kOffB + bp.slot * kBBytes + lane * (kActDigits * 128);
                    const uint32_t sfbase = ring_addr + kOffSfb + bp.slot * kSfbBytes + lane * (kActDigits * 16);
                    tma_load_2d(base, bmap, c * 128, brow, fb);
                    tma_load_2d(sfbase, sbmap, (c & ~1) * 8, brow, fb);
                }
                bp.step();
                ++issued_b;
                return true;
            };
            if (!gu && !h_ready(m)) return false;
            for (int i = 0; i < npre; ++i)
                if (!load_b(m.c0 + i)) return false;
            for (; ch < m.c1; ++ch, cp.step()) {
                if (!slot_free(sh.empty_a, cp.slot, cp.phase)) return false;
                if (lane == 0) load_codes(m, ch, cp.slot);
                ++issued;
                if (!load_b(ch)) return false;
            }
            return true;
        };
        // the tile list of a small step in registers: lane l holds tiles l and l + 32
        const bool cached = n_tiles <= 64;
        int4 tc0 = make_int4(0, 0, 0, 0), tc1 = tc0;
        if (cached) {
            if (lane < n_tiles) tc0 = a.tiles[lane];
            if (lane + 32 < n_tiles) tc1 = a.tiles[lane + 32];
        }
        auto tile_of = [&](int ti) {
            if (!cached) return a.tiles[ti];
            const int4 v = ti < 32 ? tc0 : tc1;
            return make_int4(__shfl_sync(0xffffffffu, v.x, ti & 31), __shfl_sync(0xffffffffu, v.y, ti & 31),
                             __shfl_sync(0xffffffffu, v.z, ti & 31), 0);
        };
        // The first item is the CTA's own index (no contention on the counter
        // while every CTA starts); the next index is taken from the counter
        // (offset by the grid) one item ahead, so its latency overlaps the
        // current item.  An index taken ahead was taken after the current one:
        // while a down item waits for h, the CTA holds no unstarted gate_up unit.
        int64_t it = blockIdx.x;
        for (bool first = true;; first = false) {
            if (!first) it = (int64_t)__shfl_sync(0xffffffffu, ahead, 0) + gridDim.x;
            Item m{};
            m.nsplit = 1;
            if (it < n_gu) {
                // gate_up unit: the (tile, 64-row block) over the whole K, or one
                // of its two K halves
                const int64_t u = it / nsplit;
                m.kind = 1;
                m.ti = (int)(u / rbg);
                m.rb = (int)(u % rbg);
                m.seg = (int)(it % nsplit);
                m.nsplit = nsplit;
                m.c0 = m.seg * nch_gu / nsplit;
                m.c1 = (m.seg + 1) * nch_gu / nsplit;
            } else if (it < n_gu + n_dn) {
                // down: (tile, segment, row block), so the first down items read
                // the first h blocks
                const int64_t id = it - n_gu;
                m.kind = 0;
                m.ti = (int)(id / (rbd * a.split.s_dn));
                const int rem = (int)(id % (rbd * a.split.s_dn));
                m.rb = rem % rbd;
                m.seg = rem / rbd;
                m.c0 = m.seg * a.split.l_dn;
                m.c1 = min(nch_dn, m.c0 + a.split.l_dn);
            } else {
                m.kind = -1;
                publish(m);
                break;
            }
            const int4 t = tile_of(m.ti);
            m.expert = t.x;
            m.q0 = t.y;
            m.nrows = t.z;
            ok = stream(m, first);
            if (!ok) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");   // no copy of this warp outlives the CTA
        if (*abort && lane == 0) {
            // the consumers may have stopped before the last tiles landed: wait
            // (bounded) for the tensor copies of the last code and activation positions
            volatile int never = 0;
            for (uint32_t pq = issued > (uint32_t)kCSlots ? issued - kCSlots : 0u; pq < issued; ++pq)
                (void)mbar_wait(smem_u32(&sh.full_a[pq % kCSlots]), (pq / kCSlots) & 1u, &never);
            for (uint32_t pq = issued_b > (uint32_t)kBSlots ? issued_b - kBSlots : 0u; pq < issued_b; ++pq)
                (void)mbar_wait(smem_u32(&sh.full_b[pq % kBSlots]), (pq / kBSlots) & 1u, &never);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t q = 0;
            RingPos<kBSlots> bp;
            for (int n = 0;; ++n) {
                const uint32_t islot = (uint32_t)n % kInfo;
                if (!mbar_wait(smem_u32(&sh.info_full[islot]), ((uint32_t)n / kInfo) & 1u, abort)) break;
                const Item m = get_item(sh.info[islot]);
                mbar_arrive(smem_u32(&sh.info_empty[islot]));
                if (m.kind < 0) break;
                // the previous item's accumulator has been read
                if (!mbar_wait(smem_u32(&sh.d_empty), ((uint32_t)n & 1u) ^ 1u, abort)) break;
                tc_fence_after();
                bool ok = true;
                for (int ch = m.c0; ch < m.c1; ++ch, ++q, bp.step()) {
                    const uint32_t slot = bp.slot, st = q & 1u;
                    if (!mbar_wait2(smem_u32(&sh.full_b[slot]), bp.phase, smem_u32(&sh.a_full[st]), (q >> 1) & 1u,
                                    abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bd = smem_desc_sw128(ring_addr + kOffB + slot * kBBytes);
                    // MMA t: K 64t..64t+63 of the chunk = A columns 8t..8t+7 of the
                    // stage, 32 bytes of every B row, scale word t / 2, bytes
                    // 2 (t % 2) and 2 (t % 2) + 1
#pragma unroll
                    for (uint32_t t = 0; t < 4; ++t)
                        umma_mxf4_ts(tm + kColD, tm + kColA + 32 * st + 8 * t, bd + 2 * t,
                                     idesc_mxf4(kRows, kN, 2 * (t & 1), 2 * (t & 1)),
                                     tm + kColSfa + 8 * st + 4 * (t >> 1), tm + kColSfb + 8 * st + 4 * (t >> 1),
                                     (ch != m.c0 || t != 0) ? 1u : 0u);
                    umma_commit(smem_u32(&sh.a_empty[st]));
                    umma_commit(smem_u32(&sh.empty_b[slot]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&sh.d_full));
            }
            // every MMA of this CTA has completed before its tensor memory is freed
            umma_commit(smem_u32(&sh.drain));
            volatile int never = 0;
            if (!mbar_wait(smem_u32(&sh.drain), 0u, &never)) *abort = 1;
        }
    } else {
        // ------------------------------------------------ consumers
        const int m = tid;   // weight row of the item
        const uint32_t tq = tm + ((uint32_t)(32 * warp) << 16);
        const uint32_t swz = ((uint32_t)m >> 1) & 3u;   // 64B swizzle of this code row
        uint32_t q = 0, bad_scale = 0;
        RingPos<kCSlots> cp;
        RingPos<kBSlots> bp;
        Item prev{};
        int prev_n = 0, have_prev = 0, gn = 0;   // gn: gate_up epilogues done
        for (int n = 0;; ++n) {
            const uint32_t islot = (uint32_t)n % kInfo;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.info_full[islot]), ((uint32_t)n / kInfo) & 1u, abort)))
                break;
            const Item cur = get_item(sh.info[islot]);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.info_empty[islot]));
            if (cur.kind < 0) break;
            if (have_prev && cur.kind == 0) {   // before blocking on a down item's data
                epilogue(a, sh, tq, prev, prev_n, gn, abort);
                gn += (prev.kind == 1 && prev.nsplit == 1) ? 1 : 0;
                have_prev = 0;
            }
            bool ok = true;
            for (int ch = cur.c0; ch < cur.c1; ++ch, ++q, cp.step(), bp.step()) {
                const uint32_t slot = cp.slot, st = q & 1u;
                const bool got = mbar_wait2(smem_u32(&sh.full_a[slot]), cp.phase, smem_u32(&sh.a_empty[st]),
                                            ((q >> 1) & 1u) ^ 1u, abort);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the row's 64 code bytes (16-byte unit u of the row at u ^ swz)
                const uint32_t sb = ring_addr + slot * kCodeBytes + m * 64;
                uint32_t wd[16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 v = lds_u4(sb + ((u ^ swz) << 4));
                    wd[4 * u] = v.x;
                    wd[4 * u + 1] = v.y;
                    wd[4 * u + 2] = v.z;
                    wd[4 * u + 3] = v.w;
                }
                // the chunk's two scale words of this row; then the code slot is free
                uint2 sfa = lds_u2(ring_addr + kOffSfa + slot * kSfaBytes + m * 16 + 8u * (uint32_t)(ch & 1));
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty_a[slot]));
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) expand_fp4(wd[i], r[2 * i], r[2 * i + 1]);
                if (scale_word_suspect(sfa.x) | scale_word_suspect(sfa.y)) {
                    // an invalid scale byte: that 32-element block (4 registers) counts as zero
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        uint32_t& wv = t < 4 ? sfa.x : sfa.y;
                        const int sh8 = 8 * (t & 3);
                        if (((wv >> sh8) & 0xFFu) - 1u > 251u) {
#pragma unroll
                            for (int c = 0; c < 4; ++c) r[4 * t + c] = 0u;
                            wv = (wv & ~(0xFFu << sh8)) | (127u << sh8);
                            bad_scale = 1;
                        }
                    }
                }
                // the digit rows' scale words (this quadrant's copy) come with the rows
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sh.full_b[bp.slot]), bp.phase, abort))) {
                    ok = false;
                    break;
                }
                // (lane n holds B row n's words; lanes past N repeat rows of the slot)
                const uint2 sfb = lds_u2(ring_addr + kOffSfb + bp.slot * kSfbBytes + (lane % kN) * 16 + 8u * (uint32_t)(ch & 1));
                tmem_st_stage4(tq + kColA + 32 * st, r, tq + kColSfa + 8 * st + warp, sfa.x,
                               tq + kColSfa + 8 * st + 4 + warp, sfa.y, tq + kColSfb + 8 * st, sfb.x,
                               tq + kColSfb + 8 * st + 4, sfb.y);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.a_full[st]));
                if (ch == cur.c0 && have_prev) {
                    epilogue(a, sh, tq, prev, prev_n, gn, abort);
                    gn += (prev.kind == 1 && prev.nsplit == 1) ? 1 : 0;
                    have_prev = 0;
                }
            }
            if (!ok) break;
            prev = cur;
            prev_n = n;
            have_prev = 1;
        }
        if (have_prev && !*abort) epilogue(a, sh, tq, prev, prev_n, gn, abort);
        if (bad_scale) flag_status(a.status, MOE_W2_DEV_BAD_SCALE);
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

cudaError_t launch_decode(const uint16_t* x, const int32_t* ids, const float* weights, const moe_w2_planes& w,
                          int32_t T, int32_t k, const Workspace& ws, uint16_t* y, uint32_t* status, cudaStream_t s,
                          const PhaseEvents& ev)
{
    (void)x;
    const int32_t E = w.num_experts, H = w.hidden, I = w.inter;
    const int64_t P = (int64_t)T * k;
    constexpr int kDyn = kRingBytes + 1024;
    static bool ready[kMaxDevices];
    static int occ_of[kMaxDevices];
    int dev = 0;
    cudaError_t e0 = once_per_device(ready, dev, [&](int d) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn);
        if (e != cudaSuccess) return e;
        // all of the unified L1 as shared memory: four CTAs per SM (their tensor
        // memory, 4 x 128 columns, fills the SM's)
        e = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        // CTAs per SM from this kernel's own resources (the occupancy query
        // reports one CTA per SM for any kernel that allocates tensor memory,
        // although four 128-column CTAs do run side by side)
        cudaFuncAttributes fa{};
        if ((e = cudaFuncGetAttributes(&fa, decode_layer_kernel)) != cudaSuccess) return e;
        int smem_sm = 0, resv = 0, regs_sm = 0;
        if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, d)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, d)) != cudaSuccess)
            return e;
        const int by_smem = smem_sm / (kDyn + (int)fa.sharedSizeBytes + resv);
        const int regs_cta = ((fa.numRegs * 32 + 255) / 256) * 256 * (kThreads / 32);
        const int by_regs = regs_cta > 0 ? regs_sm / regs_cta : 1;
        occ_of[d] = std::max(1, std::min({by_smem, by_regs, (int)(512 / kTmemCols)}));
        return cudaSuccess;
    });
    if (e0 != cudaSuccess) return e0;
    const int occ = occ_of[dev];
    const int64_t mt = max_tiles(P, E, true);

    LayerArgs a{};
    a.H = H;
    a.I = I;
    a.T = T;
    a.k = k;
    a.E = E;
    a.split = ws.split;
    a.P = P;
    a.tiles = ws.tiles;
    a.tile_count = ws.tile_count;
    a.sorted = ws.sorted;
    a.weights = weights;
    a.xd = ws.xd;
    a.sxd = ws.sxd;
    a.hd = ws.hd;
    a.shd = ws.shd;
    a.stage = ws.stage;
    a.h_flag = ws.counters;                    // zeroed by the permutation kernel
    a.gu_cnt = a.h_flag + mt * (I / 64);
    a.queue = a.gu_cnt + mt * (I / 64);
    a.gu_part = ws.gu_part;
    a.ids = ids;
    a.dep = dependency_wait();
    a.status = status;

    // code tiles: 64 bytes (256 codes) x 128 rows, 64B-swizzled; gate_up as a
    // 3-D box {64 bytes, 64 rows, 2 planes} over the w13 plane seen as 2E planes
    // (gate, up) of I rows, down as a 2-D box of 128 rows
    CUtensorMap gu_map, dn_map;
    cudaError_t e = make_tmap_3d_u8(&gu_map, w.w13_codes, 2 * (int64_t)E, I, H / 4, 64, 64, 2, 64);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_2d(&dn_map, w.w2_codes, false, (int64_t)E * H, I / 4, 64, 128, 64)) != cudaSuccess) return e;
    // scale groups: 16 bytes (2 chunks) x 64 rows (gate_up) or x 128 rows (down);
    // rows of H/32 and I/32 bytes are multiples of 16 (H, I multiples of 512)
    CUtensorMap gu_sf_map, dn_sf_map;
    if ((e = make_tmap_3d_u8(&gu_sf_map, w.w13_scales, 2 * (int64_t)E, I, H / 32, 16, 64, 2, 0)) != cudaSuccess)
        return e;
    if ((e = make_tmap_2d(&dn_sf_map, w.w2_scales, false, (int64_t)E * H, I / 32, 16, 128, 0)) != cudaSuccess)
        return e;

    // activation digit rows: boxes of one pair's 8 rows x 128 bytes (256 K),
    // 128B-swizzled as the UMMA B operand, and their 16-byte scale groups
    CUtensorMap xd_map, sxd_map, hd_map, shd_map;
    if ((e = make_tmap_2d(&xd_map, ws.xd, false, (int64_t)kActDigits * T, H / 2, 128, kActDigits, 128)) != cudaSuccess ||
        (e = make_tmap_2d(&sxd_map, ws.sxd, false, (int64_t)kActDigits * T, H / 32, 16, kActDigits, 0)) != cudaSuccess ||
        (e = make_tmap_2d(&hd_map, ws.hd, false, (int64_t)kActDigits * P, I / 2, 128, kActDigits, 128)) != cudaSuccess ||
        (e = make_tmap_2d(&shd_map, ws.shd, false, (int64_t)kActDigits * P, I / 32, 16, kActDigits, 0)) != cudaSuccess)
        return e;

    const int grid = sm_count() * occ;
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
    if ((e = cudaLaunchKernelEx(&cfg, decode_layer_kernel, gu_map, dn_map, gu_sf_map, dn_sf_map, xd_map, sxd_map,
                                hd_map, shd_map, a)) != cudaSuccess)
        return e;
    if ((e = ev.record(2, s)) != cudaSuccess) return e;
    // y = the slots of every token summed over j and the K segments of down
    return launch_combine(ws.stage, ids, T, k, E, H, a.split.s_dn, P * H, true, y, s);
}

}  // namespace moe_w2
