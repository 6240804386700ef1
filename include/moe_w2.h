/*
 * moe_w2 — routed-expert MoE layer with 2-bit sign-symmetric expert weights,
 * for NVIDIA GB300 (sm_103a).  C ABI: plain pointers, sizes and a CUDA stream.
 *
 * What the library computes (vLLM-Moet pages):
 *   - "vLLM-Moet wiki", section "2-bit expert planes": routed experts stored as
 *     2-bit codes from the sign-symmetric codebook {-4,-1,1,4};
 *   - "vLLM-Moet wiki", section "The kernels": the 2-bit MoE GEMM (in-register
 *     code expansion feeding tensor cores), deterministic, graph-capture safe;
 *   - "The v0.24.0 port", section "Our hooks": moe_w2_forward in the quant
 *     method's apply hook; the modelopt NVFP4 loader that dequantizes
 *     e2m1 x e4m3 block-16 x scale_2 exactly in f64 and re-quantizes to the
 *     codebook with UE8M0 block-32 scales absorbing scale_2; codes + UE8M0
 *     scales as four sections per expert slot; the deterministic unpermute
 *     (bijective per-pair placement + fixed-order sum over top_k).
 *
 * Plane format (the four sections per expert):
 *   w13_codes  uint8 [E][2I][H/4]   rows 0..I-1 = gate, rows I..2I-1 = up
 *   w13_scales uint8 [E][2I][H/32]
 *   w2_codes   uint8 [E][H][I/4]    down projection
 *   w2_scales  uint8 [E][H][I/32]
 *   Weight (r, kk) = code_value(c) * 2^(s - 127) with
 *     c = (codes[r][kk/4] >> (2*(kk%4))) & 3, code_value = {+1, +4, -1, -4}[c]
 *     (c = sign<<1 | magnitude), s = scales[r][kk/32] in [1, 252].
 *
 * Conventions for every entry point:
 *   - Every buffer is owned by the caller and lives in device memory unless
 *     stated otherwise (moe_w2_forward_noalloc's scratch is the library's).
 *     The library allocates nothing, frees nothing and never synchronises:
 *     work is enqueued on `stream` (a cudaStream_t, NULL =
 *     the legacy default stream) and completes asynchronously.  No entry point
 *     reads a device value on the host, so all of them can be captured in a
 *     CUDA graph (this remark does not extend to moe_w2_forward_noalloc).
 *   - Host-side argument checks return a status code and enqueue nothing.
 *   - Device-side input errors never trap: they OR a bit into *dev_status
 *     (a device uint32 the caller zeroes and reads back; NULL = do not report)
 *     and the offending contribution is replaced as documented per bit.
 *   - Results are deterministic: identical inputs give bitwise identical outputs.
 *   - Host threads may call the entry points concurrently, on any device and
 *     stream, as long as concurrent calls do not share a workspace or an
 *     output buffer.  The one-time set-up of each kernel on each device
 *     (shared-memory attributes, occupancy) happens on the first call there,
 *     serialised by a lock inside the library.
 *   - Requires a device of compute capability 10.3 (GB300).
 */
#ifndef MOE_W2_H
#define MOE_W2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_W2_OK = 0,
    MOE_W2_ERR_INVALID_ARG = 1,       /* null pointer, negative size, top_k or E out of range */
    MOE_W2_ERR_UNSUPPORTED_SHAPE = 2, /* H or I not a multiple of 256, K not a multiple of 32, too many pairs */
    MOE_W2_ERR_WORKSPACE = 3,         /* workspace smaller than moe_w2_forward_workspace_size() */
    MOE_W2_ERR_CUDA = 4,              /* a CUDA call or kernel launch failed (cudaGetLastError) */
    MOE_W2_ERR_DEVICE = 5             /* the current device is not compute capability 10.3 */
} moe_w2_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define MOE_W2_DEV_BAD_EXPERT_ID 1u   /* topk id outside [0,E): that pair contributes 0 */
#define MOE_W2_DEV_BAD_SCALE 2u       /* UE8M0 byte outside [1,252] in a plane: that block counts as 0 */
#define MOE_W2_DEV_BAD_NVFP4 4u       /* requant input (NVFP4 or FP8): e4m3 NaN in a block, or its scale_2 /
                                         block scale not a positive finite number: the block's codes are
                                         0x00 and its scale byte 0 */
#define MOE_W2_DEV_PIPELINE_TIMEOUT 0x80000000u
                                      /* a kernel's internal wait (a pipeline barrier, or a hand-over
                                         between two phases of the layer) passed its limit of about
                                         two seconds: the kernel stopped, freed its tensor memory and
                                         returned, and the outputs of that call are not valid.  Never
                                         expected; the stream and the context stay usable. */

/* Limits checked on the host. */
#define MOE_W2_MAX_EXPERTS 1024
#define MOE_W2_MAX_TOP_K 16
#define MOE_W2_MAX_PAIRS (1 << 21)    /* T * top_k */
#define MOE_W2_MAX_ROUTED_EXPERTS (1 << 20)   /* length of a residency table (moe_w2_forward_cached) */
#define MOE_W2_DECODE_MAX_TOKENS 64   /* T <= 64 runs the decode kernels, larger T the prefill kernels */

/* Device pointers to one layer's planes (layout above). */
typedef struct {
    const uint8_t *w13_codes;
    const uint8_t *w13_scales;
    const uint8_t *w2_codes;
    const uint8_t *w2_scales;
    int32_t num_experts; /* E */
    int32_t hidden;      /* H, multiple of 256 */
    int32_t inter;       /* I, multiple of 256 */
} moe_w2_planes;

/* Bytes of device workspace moe_w2_forward needs for these sizes (0 if the sizes
 * are invalid).  The workspace holds the permutation, the expert-sorted and
 * re-laid-out activations, the SiLU(gate)*up intermediate h (bf16, P x I), the
 * fp32 per-pair staging of the deterministic combine (P x H) and the decode
 * path's per-row-block completion counters.  Its contents need no
 * initialisation: every call writes each part before reading it. */
size_t moe_w2_forward_workspace_size(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I);

/* Which kernels moe_w2_forward runs for these sizes (host only, no device
 * access): MOE_W2_PATH_DECODE_STREAM for decode steps (T <= 64) of at most 16
 * pairs with H and I multiples of 512 (the stream-K tcgen05 block-scaled
 * kernel, one CTA per SM, y summed in the same launch);
 * MOE_W2_PATH_DECODE_MMA for decode steps with H or I not a multiple of 512
 * (the bf16 mma.sync kernel); MOE_W2_PATH_DECODE_BLOCK_SCALED for the other
 * decode steps (the tcgen05 block-scaled kernel and its combine);
 * MOE_W2_PATH_PREFILL for T > 64 (the
 * gather, the two tcgen05 GEMMs and the combine); MOE_W2_PATH_NONE when the
 * sizes are invalid (moe_w2_forward_workspace_size would return 0) or T = 0.
 * The pages describe no such entry point: it keeps the dispatch rule in one
 * place for bindings and benchmarks. */
#define MOE_W2_PATH_NONE 0
#define MOE_W2_PATH_DECODE_MMA 1
#define MOE_W2_PATH_DECODE_BLOCK_SCALED 2
#define MOE_W2_PATH_PREFILL 3
#define MOE_W2_PATH_DECODE_STREAM 4
int moe_w2_forward_path(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I);

/*
 * Routing permutation ("The v0.24.0 port", "Our hooks", deterministic
 * unpermute bullet: valid sorted ids are a permutation of token*top_k+j).
 *   topk_ids       int32 [T][top_k]   expert of pair p = t*top_k + j
 *   sorted_pairs   int32 [T*top_k]    pair ids grouped by expert: expert 0's pairs
 *                                     in increasing p, then expert 1's, ...; pairs
 *                                     with an id outside [0,E) come last (in
 *                                     increasing p) and set MOE_W2_DEV_BAD_EXPERT_ID
 *   inv_pairs      int32 [T*top_k]    inv_pairs[sorted_pairs[q]] = q
 *   expert_offsets int32 [E+1]        first slot of each expert; [E] = valid pairs
 * T = 0 is a no-op.  Bit-exact and deterministic (a stable counting sort).
 */
moe_w2_status moe_w2_permute(const int32_t *topk_ids, int32_t T, int32_t top_k, int32_t E,
                             int32_t *sorted_pairs, int32_t *inv_pairs, int32_t *expert_offsets,
                             uint32_t *dev_status, void *stream);

/*
 * Routed-expert forward ("vLLM-Moet wiki", "The kernels"; "The v0.24.0 port",
 * "Our hooks"): for every token t and slot j with e = topk_ids[t][j],
 *     g = W_gate[e] x_t,  u = W_up[e] x_t            (fp32 accumulation)
 *     h = bf16(SiLU(g) * u)
 *     y_t = bf16( sum_j topk_weights[t][j] * (W_down[e] h) )   (fp32)
 *   x_bf16        bf16 [T][H]
 *   topk_ids      int32 [T][top_k]
 *   topk_weights  float [T][top_k]
 *   w             host pointer to the plane pointers (read during the call only)
 *   y_bf16        bf16 [T][H] (written; may not alias x)
 *   workspace     device buffer of at least moe_w2_forward_workspace_size() bytes,
 *                 256-byte aligned, used by this call until it completes on `stream`
 * x_bf16, y_bf16 and the four plane pointers must be 16-byte aligned
 * (MOE_W2_ERR_INVALID_ARG otherwise).
 * T = 0 is a no-op.  Pairs with an id outside [0,E) contribute 0
 * (MOE_W2_DEV_BAD_EXPERT_ID); blocks with a UE8M0 byte outside [1,252] count
 * as 0 (MOE_W2_DEV_BAD_SCALE).  T <= 64 uses the decode kernels, which stream
 * the planes of every active expert once per step: steps of more than 16 pairs
 * with H and I multiples of 512 a block-scaled tcgen05 kernel (codes expanded
 * to packed e2m1, activations as eight packed e2m1 digit rows, both scaled by
 * UE8M0 bytes per 32 elements), the rest a bf16 mma.sync kernel; larger T the
 * prefill kernels (TMA + tcgen05 with accumulators in tensor memory).
 */
moe_w2_status moe_w2_forward(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                             const moe_w2_planes *w, int32_t T, int32_t top_k, void *y_bf16,
                             void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream);

/*
 * moe_w2_forward with phase events, for profiling: identical work and results.
 *   phase_events  host array of 4 cudaEvent_t (or NULL entries); event i is
 *                 recorded on `stream` before phase i: 0 = before the
 *                 permutation, 1 = before the gate_up kernel(s), 2 = before the
 *                 down kernel(s), 3 = after the last kernel.  On the prefill
 *                 path the gather is part of phase 0..1 and the combine of 2..3.
 *                 On the decode path one kernel runs gate_up and down (1..2)
 *                 and 2..3 is the combine kernel (empty for the mma.sync
 *                 kernel, which sums the slots itself).
 * cudaEventRecord failures return MOE_W2_ERR_CUDA.
 */
moe_w2_status moe_w2_forward_traced(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                                    const moe_w2_planes *w, int32_t T, int32_t top_k, void *y_bf16,
                                    void *workspace, size_t workspace_bytes, uint32_t *dev_status,
                                    void *stream, void *const *phase_events);

/*
 * moe_w2_forward without a caller-supplied workspace, for callers that cannot
 * allocate device memory where they run the layer (an allocator that may not
 * grow, device memory already handed out in full, or a point where an
 * allocation would synchronise the device).  The pages describe no such entry point:
 * it is an interface addition of this library.
 * Same arguments, results and status codes as moe_w2_forward, minus
 * workspace and workspace_bytes: the scratch is a device array of
 * MOE_W2_NOALLOC_WORKSPACE_BYTES that the library owns; each GPU that loads
 * the library's device code holds it until the process exits.
 *   - Sizes whose moe_w2_forward_workspace_size() exceeds
 *     MOE_W2_NOALLOC_WORKSPACE_BYTES return MOE_W2_ERR_WORKSPACE and enqueue
 *     nothing (at H=6144, I=2048, E=256, top_k=8 that is T > 28).
 *   - The first call in each CUDA context (normally a device's primary
 *     context) checks the device and looks up the array's address
 *     (cudaGetSymbolAddress, with that device current), then keeps it for
 *     that context; make that first call before any stream capture starts.
 *     cudaDeviceReset destroys the context and the array with it: the next
 *     call recognises the new context and looks the address up again.
 *   - Every call on a device uses the same array, so calls that may run at
 *     the same time race: order them (e.g. issue them on one stream).
 *   - Nothing in the array needs to start at zero, and a call's results do
 *     not depend on what earlier calls left in it: they are bitwise identical
 *     to moe_w2_forward's on the same inputs.
 */
#define MOE_W2_NOALLOC_WORKSPACE_BYTES (8u << 20)
moe_w2_status moe_w2_forward_noalloc(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                                     const moe_w2_planes *w, int32_t T, int32_t top_k, void *y_bf16,
                                     uint32_t *dev_status, void *stream);

/*
 * moe_w2_forward behind an expert cache ("vLLM-Moet wiki", BASE-cache
 * paragraph; "The v0.24.0 port", "Our hooks", BASE-cache bullet): w holds
 * num_slots = w->num_experts resident experts, and a residency table says
 * where each routed expert is.
 *   slot_of_expert      int32 [num_routed_experts] (device): slot in
 *                       [0, w->num_experts) of each routed expert id, or any
 *                       negative value when that expert is not resident
 *   num_routed_experts  length of the table, 1 .. MOE_W2_MAX_ROUTED_EXPERTS;
 *                       topk_ids are routed ids in [0, num_routed_experts)
 *   miss_counter        device uint32 (NULL = do not count): the call adds the
 *                       number of pairs whose expert is not resident
 *   workspace           at least moe_w2_forward_cached_workspace_size() bytes
 * A pair whose expert is not resident contributes 0 to y and sets no status
 * bit: its step can be replayed once the caller has loaded the missing experts.
 * A routed id outside [0, num_routed_experts) or a table entry >= num_slots is
 * an invalid id (contributes 0, MOE_W2_DEV_BAD_EXPERT_ID).  Every other
 * argument, check and result is as for moe_w2_forward; in particular y for a
 * step with every expert resident is bitwise identical to moe_w2_forward's
 * with the same experts' planes at any slots, since each pair's result and the
 * fixed j-order sum do not depend on where its expert sits.
 */
size_t moe_w2_forward_cached_workspace_size(int32_t T, int32_t top_k, int32_t num_slots, int32_t H, int32_t I);
moe_w2_status moe_w2_forward_cached(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                                    const moe_w2_planes *w, const int32_t *slot_of_expert,
                                    int32_t num_routed_experts, int32_t T, int32_t top_k, void *y_bf16,
                                    void *workspace, size_t workspace_bytes, uint32_t *miss_counter,
                                    uint32_t *dev_status, void *stream);

/*
 * Load-time re-quantizer ("The v0.24.0 port", "Our hooks", modelopt.py
 * bullet): modelopt NVFP4 tensors -> 2-bit planes.
 *   e2m1     uint8 [n][rows][K/2]   two e2m1 nibbles per byte, low nibble = even element
 *   e4m3     uint8 [n][rows][K/16]  e4m3fn block-16 scales
 *   scale_2  float [n]              per-tensor scale (device memory)
 *   codes    uint8 [n][rows][K/4]   output codes (plane format above)
 *   ue8m0    uint8 [n][rows][K/32]  output UE8M0 bytes, s = u + 127
 * Per block of 32 consecutive elements x_i = e2m1_i * e4m3 * scale_2 (exact),
 * the output is the u in [-126,125] minimising sum_i (x_i - v_i 2^u)^2 exactly,
 * with every v_i the nearest of {-4,-1,1,4} (|x| > 2.5*2^u -> magnitude 4, else
 * 1; the code's sign is x's sign bit, so -0 -> -1); ties between scales go to
 * the smaller u.  Bit-exact.  Invalid blocks: see MOE_W2_DEV_BAD_NVFP4.
 * K must be a multiple of 32; n*rows*K/32 blocks must fit in int64.
 */
moe_w2_status moe_w2_requant(const uint8_t *e2m1, const uint8_t *e4m3, const float *scale_2,
                             int64_t n, int64_t rows, int64_t K, uint8_t *codes, uint8_t *ue8m0,
                             uint32_t *dev_status, void *stream);

/*
 * Option bits of the FP4 loaders (moe_w2_requant_ex, moe_w2_requant_mxfp4).
 * MOE_W2_REQUANT_BALANCE_ZERO_SIGNS ("vLLM-Moet wiki", the Kimi-K2.7
 * paragraph: an export that writes every exact zero as +0 would bias the
 * codes): the elements of a block that are exactly zero get the signs
 * +,-,+,- ... in element order (the first zero of the block +1, the second -1,
 * ...) instead of their stored sign bits.  A zero is at magnitude 1 for every
 * scale, so the scale byte and every other code are unchanged.  Other bits are
 * reserved: a call with one of them set returns MOE_W2_ERR_INVALID_ARG.
 */
#define MOE_W2_REQUANT_BALANCE_ZERO_SIGNS 1u

/* moe_w2_requant with option bits (options = 0: identical to moe_w2_requant). */
moe_w2_status moe_w2_requant_ex(const uint8_t *e2m1, const uint8_t *e4m3, const float *scale_2,
                                int64_t n, int64_t rows, int64_t K, uint32_t options, uint8_t *codes,
                                uint8_t *ue8m0, uint32_t *dev_status, void *stream);

/*
 * Load-time re-quantizer for MXFP4 checkpoints ("The v0.24.0 port", "Our
 * hooks", mxfp4.py bullet; "vLLM-Moet wiki": FP4 experts load by a codes
 * remap): e2m1 elements with one UE8M0 scale byte per 32 -> 2-bit planes.
 *   e2m1    uint8 [n][rows][K/2]    two nibbles per byte, low nibble = even element
 *   scales  uint8 [n][rows][K/32]   UE8M0 bytes s, element value e2m1 * 2^(s-127)
 *   codes   uint8 [n][rows][K/4]    output codes (plane format above)
 *   ue8m0   uint8 [n][rows][K/32]   output UE8M0 bytes
 *   options MOE_W2_REQUANT_BALANCE_ZERO_SIGNS or 0
 * Same rule as moe_w2_requant (least squared error over u in [-126,125],
 * nearest code, ties to magnitude 1 and to the smaller u, -0 -> -1).  Because
 * the input scale is a power of two, the codes depend only on the block's
 * e2m1 codes and the output byte is the input byte plus a shift that also
 * depends only on them, except where the exponent range [-126,125] cuts the
 * search.  Bit-exact.  Scale byte 255 (NaN) makes the block invalid: codes
 * 0x00, scale byte 0, MOE_W2_DEV_BAD_NVFP4.  K must be a multiple of 32; e2m1
 * 16-byte aligned, codes 8-byte aligned.
 */
moe_w2_status moe_w2_requant_mxfp4(const uint8_t *e2m1, const uint8_t *scales, int64_t n, int64_t rows, int64_t K,
                                   uint32_t options, uint8_t *codes, uint8_t *ue8m0, uint32_t *dev_status,
                                   void *stream);

/*
 * Test hook for the pipeline-timeout report; the pages describe no such entry
 * point.  With enable != 0, every later moe_w2_forward call in this process
 * (any thread, any device) that runs a decode kernel makes that kernel's
 * cross-CTA dependency wait (a down item waiting for the h it reads)
 * unsatisfiable with a limit of about 0.1 ms: the wait gives up, the kernel
 * stops, frees its tensor memory and returns with MOE_W2_DEV_PIPELINE_TIMEOUT
 * set in *dev_status, and y is not valid.  Nothing faults or hangs, and the
 * stream and context stay usable.  enable = 0 (the default) restores normal
 * operation for the calls that follow.  Always returns MOE_W2_OK.
 */
moe_w2_status moe_w2_debug_force_pipeline_timeout(int32_t enable);

/*
 * Kernel choice for the smallest decode steps (at most 16 pairs, H and I
 * multiples of 512 and at most 7168).  With enable != 0 (the default), every
 * later call in this process (any thread, any device) runs such steps on the
 * stream-K kernel (MOE_W2_PATH_DECODE_STREAM: one CTA per SM streams every
 * active expert's planes, multiplied on the tensor cores in block-scaled FP4);
 * with enable = 0 they run on the mma.sync kernel (MOE_W2_PATH_DECODE_MMA).
 * Both compute the same layer ("vLLM-Moet wiki", section "The kernels") within
 * the same error bound.  The workspace a step needs depends on the choice
 * (moe_w2_forward_workspace_size answers for the current one; a forward given
 * less returns MOE_W2_ERR_WORKSPACE).  Always returns MOE_W2_OK.
 */
moe_w2_status moe_w2_set_decode_stream(int32_t enable);

/*
 * Load-time re-quantizer for FP8 block-quantised checkpoints ("The v0.24.0
 * port", "Our hooks", fp8.py bullet): fp8 weights with f32 block-128 scales ->
 * 2-bit planes.
 *   w8      uint8 [n][rows][K]                       e4m3fn bytes
 *   scales  float [n][ceil(rows/128)][ceil(K/128)]   one scale per 128 x 128 block
 *                                                    (row block r/128, column block k/128)
 *   codes   uint8 [n][rows][K/4]    output codes (plane format above)
 *   ue8m0   uint8 [n][rows][K/32]   output UE8M0 bytes, s = u + 127
 * Per block of 32 consecutive elements x_i = e4m3_i * S (exact), the output
 * follows the same rule as moe_w2_requant (least squared error over u in
 * [-126,125], nearest code, ties to magnitude 1 and to the smaller u, -0 -> -1).
 * Bit-exact.  A block with an e4m3 NaN, or whose scale is not a positive finite
 * number, gets codes 0x00 and scale byte 0 and sets MOE_W2_DEV_BAD_NVFP4.
 * K must be a multiple of 32; w8 16-byte aligned, codes 8-byte aligned.
 */
moe_w2_status moe_w2_requant_fp8(const uint8_t *w8, const float *scales, int64_t n, int64_t rows, int64_t K,
                                 uint8_t *codes, uint8_t *ue8m0, uint32_t *dev_status, void *stream);

/*
 * The FP4 layer ("vLLM-Moet wiki", "The kernels" and "FP4 recovery": moe_w4_mm,
 * the same MoE forward over the NVFP4 experts, at twice the 2-bit plane bytes):
 * every weight is e2m1 x e4m3 (one scale per 16 consecutive K elements of a row)
 * x scale_2 (one per tensor: gate, up and down of each expert), taken exactly.
 *   w13_e2m1     uint8 [E][2I][H/2]   two nibbles per byte, low nibble = even element;
 *                                     rows 0..I-1 gate, I..2I-1 up
 *   w13_e4m3     uint8 [E][2I][H/16]  e4m3fn block scales
 *   w13_scale_2  float [E][2]         gate's and up's scale_2 (device memory)
 *   w2_e2m1      uint8 [E][H][I/2]
 *   w2_e4m3      uint8 [E][H][I/16]
 *   w2_scale_2   float [E]            down's scale_2 (device memory)
 * These are the modelopt NVFP4 tensors as moe_w2_requant takes them, laid out
 * per expert like the 2-bit planes.
 */
typedef struct {
    const uint8_t *w13_e2m1;
    const uint8_t *w13_e4m3;
    const float *w13_scale_2;
    const uint8_t *w2_e2m1;
    const uint8_t *w2_e4m3;
    const float *w2_scale_2;
    int32_t num_experts; /* E */
    int32_t hidden;      /* H, multiple of 256 */
    int32_t inter;       /* I, multiple of 256 */
} moe_w4_planes;

/* Bytes of device workspace moe_w4_forward needs (0 if the sizes are invalid). */
size_t moe_w4_forward_workspace_size(int32_t T, int32_t top_k, int32_t E, int32_t H, int32_t I);

/*
 * moe_w2_forward over NVFP4 experts: for every token t and slot j with
 * e = topk_ids[t][j], g = W_gate[e] x_t, u = W_up[e] x_t, h = bf16(SiLU(g) u),
 * y_t = bf16(sum_j topk_weights[t][j] (W_down[e] h)), with each W the exact
 * NVFP4 value above (e2m1 x e4m3 products are exact in bf16; scale_2
 * multiplies the fp32 accumulations).  Arguments, alignment, checks, status
 * bits and determinism as for moe_w2_forward; the four byte planes and the two
 * scale_2 arrays must be 16- and 4-byte aligned.  An e4m3 NaN scale makes its
 * 16 weights count as 0 and sets MOE_W2_DEV_BAD_SCALE; scale_2 is used as
 * given (a non-finite one gives non-finite outputs).  T <= 64 runs the bf16
 * mma.sync decode kernel (every active expert's planes streamed once per
 * step), larger T the TMA + tcgen05 prefill kernels.
 */
moe_w2_status moe_w4_forward(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                             const moe_w4_planes *w, int32_t T, int32_t top_k, void *y_bf16,
                             void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream);

/* moe_w4_forward with the four phase events of moe_w2_forward_traced (profiling). */
moe_w2_status moe_w4_forward_traced(const void *x_bf16, const int32_t *topk_ids, const float *topk_weights,
                                    const moe_w4_planes *w, int32_t T, int32_t top_k, void *y_bf16,
                                    void *workspace, size_t workspace_bytes, uint32_t *dev_status, void *stream,
                                    void *const *phase_events);

/* Human-readable name of a status code (static string). */
const char *moe_w2_status_string(moe_w2_status s);

/* Library version, (major << 16) | minor. */
int moe_w2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W2_H */
