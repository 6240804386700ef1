"""Seeded synthetic inputs for the 2-bit MoE layer and for the NVFP4 re-quantizer.

This module only draws random numbers and lays them out in the storage formats.
It holds none of the layer's arithmetic (no dequantisation, no re-quantisation,
no permutation, no expert math), so both the CUDA path and the CPU oracle can be
fed from it without sharing any of the method.

Workloads (shapes follow the models named on the vLLM-Moet pages: GLM-5.x and
DeepSeek-V4-Flash experts, top-8 routing, hidden 6144/4096, expert intermediate
2048; page "vLLM-Moet wiki", section "The kernels", and page "The v0.24.0 port",
section "Our hooks"):

  tiny            H=512  I=256  E=8   top-2 T=4     UE8M0 exponents in [-9,-6]  router logits
  decode_t1       H=6144 I=2048 E=256 top-8 T=1     exponents in [-10,-6]       Zipf(1.1) routing
  decode_t32      H=6144 I=2048 E=256 top-8 T=32    exponents in [-10,-6]       Zipf(1.1) routing
  prefill_t8192   H=4096 I=2048 E=256 top-8 T=8192  exponents in [-10,-6]       router logits
  requant_256     256 experts of NVFP4 gate/up [2048x6144] and down [6144x2048]
  decode_t1_e32, prefill_t1024_e32: the decode_t1 / prefill_t8192 layers over 32 experts
                  (same per-launch kernel work; small enough for multi-pass profiling)

Recipe (all numpy PCG64 via ``default_rng(seed)``):
  * activations: standard normal fp32, rounded to bf16 (round to nearest even);
    returned as the uint16 bit pattern.
  * code planes: uniform random bytes (raw PCG64 words read as little-endian
    bytes; every 2-bit field is then uniform over the four codes and
    independent); UE8M0 scale bytes 127 + integers(lo, hi+1) drawn as uint8.
  * router "logits": standard normal (T, E) fp32, top-k by value with ties to the
    lower id, weights = softmax over the k selected logits.
  * router "zipf": expert popularity p_r proportional to r^-1.1 (r = 1..E), rank r
    mapped to expert id perm[r-1] for perm = rng.permutation(E); each token draws
    k distinct experts with those probabilities; weights = softmax of k standard
    normal logits.
  * NVFP4 tensors: e2m1 nibbles uniform over all 16 codes (uniform random bytes,
    low nibble = even element), e4m3 block-16 scales 2^U(-6, 2) rounded to the
    nearest e4m3fn value (ties to even mantissa), scale_2 = 2^-8 per tensor.
  * FP8 block-quantised tensors (the fp8 loader's input): e4m3fn bytes uniform
    over the 254 non-NaN codes, one f32 scale per 128 x 128 block drawn
    log-uniform, 2^U(-14, -8), rounded to f32 (a general mantissa).
  * wide-range activations (parity cases for activations with a large dynamic
    range inside a 32-element block, as real LLM activations have):
    "outlier": standard normal, then in every aligned block of 32 one element
    at a uniform position multiplied by 2^e, e uniform in [lo, hi];
    "zeros": every element zero with probability 1/2, and every other block
    multiplied by 2^10 (blocks mixing exact zeros with large values);
    "both": the two applied one after the other.
  * wide-range h: in every expert, for each aligned block of 32 rows of the
    gate and up halves, one row (uniform position, the same row in gate and up)
    gets its UE8M0 exponents raised by `boost`, so that h = SiLU(g) * u has one
    element per 32 that is about 2^(2 boost) times the others.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    hidden: int          # H
    inter: int           # I
    num_experts: int     # E
    top_k: int           # k
    tokens: int          # T
    exp_lo: int          # UE8M0 exponent range of the code planes
    exp_hi: int
    routing: str         # "logits" or "zipf"
    seed: int

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k

    @property
    def plane_bytes_per_expert(self) -> int:
        H, I = self.hidden, self.inter
        return 2 * I * (H // 4) + 2 * I * (H // 32) + H * (I // 4) + H * (I // 32)


@dataclasses.dataclass(frozen=True)
class RequantConfig:
    name: str
    num_experts: int
    inter: int
    hidden: int
    seed: int


CONFIGS = {
    "tiny": LayerConfig("tiny", 512, 256, 8, 2, 4, -9, -6, "logits", 0),
    "decode_t1": LayerConfig("decode_t1", 6144, 2048, 256, 8, 1, -10, -6, "zipf", 1),
    "decode_t32": LayerConfig("decode_t32", 6144, 2048, 256, 8, 32, -10, -6, "zipf", 2),
    "prefill_t8192": LayerConfig("prefill_t8192", 4096, 2048, 256, 8, 8192, -10, -6, "logits", 3),
    # Small cases with the same per-launch kernel work, for multi-pass profiler captures:
    # a T=1 step streams 8 experts' planes whatever E is, and T=1024 over 32 experts gives
    # the same 256 pairs per expert as T=8192 over 256 experts (an eighth of the tiles).
    "decode_t1_e32": LayerConfig("decode_t1_e32", 6144, 2048, 32, 8, 1, -10, -6, "zipf", 5),
    "prefill_t1024_e32": LayerConfig("prefill_t1024_e32", 4096, 2048, 32, 8, 1024, -10, -6, "logits", 6),
}
REQUANT = RequantConfig("requant_256", 256, 2048, 6144, 4)
# Re-quantizer workloads by name: experts drawn from REQUANT (None = all).  requant_16
# is the first 16 experts of the same draw (each expert has its own child seed): the
# same per-block kernel work on 1/16 of the data, for multi-pass profiler captures.
REQUANT_CASES = {"requant_256": None, "requant_16": 16}
# FP8 block-128 loader workloads: experts of gate/up [I][H] x 2 and down [H][I]
REQUANT_FP8_CASES = {"requant_fp8_16": 16}
# The FP4 layer (NVFP4 experts): a decode step and a prefill step of the 2-bit
# layers' shapes over 64 experts (a step of T = 1 streams 8 experts whatever E is)
W4_CONFIGS = {
    "w4_decode_t1_e64": LayerConfig("w4_decode_t1_e64", 6144, 2048, 64, 8, 1, -10, -6, "zipf", 21),
    "w4_prefill_t8192_e64": LayerConfig("w4_prefill_t8192_e64", 4096, 2048, 64, 8, 8192, -10, -6, "logits", 22),
}
# MXFP4 loader workloads (e2m1 with UE8M0 block-32 scales), same expert shapes
REQUANT_MXFP4_CASES = {"requant_mxfp4_16": 16}


def rng_for(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def random_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform random bytes: raw 64-bit PCG64 outputs read as little-endian bytes."""
    n = int(np.prod(shape))
    words = rng.bit_generator.random_raw((n + 7) // 8)
    return words.view(np.uint8)[:n].reshape(shape)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def activations(rng: np.random.Generator, T: int, H: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))


def ue8m0_bytes(rng: np.random.Generator, shape, exp_lo: int, exp_hi: int) -> np.ndarray:
    """UE8M0 bytes 127 + e with e uniform over [exp_lo, exp_hi]."""
    return rng.integers(127 + exp_lo, 127 + exp_hi + 1, size=shape, dtype=np.uint8)


def code_planes(rng: np.random.Generator, E: int, H: int, I: int, exp_lo: int, exp_hi: int):
    """Random 2-bit expert planes: codes uniform over the four codes, exponents uniform."""
    w13_codes = random_bytes(rng, (E, 2 * I, H // 4))
    w13_scales = ue8m0_bytes(rng, (E, 2 * I, H // 32), exp_lo, exp_hi)
    w2_codes = random_bytes(rng, (E, H, I // 4))
    w2_scales = ue8m0_bytes(rng, (E, H, I // 32), exp_lo, exp_hi)
    return {"w13_codes": w13_codes, "w13_scales": w13_scales,
            "w2_codes": w2_codes, "w2_scales": w2_scales}


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def wide_range_activations(rng: np.random.Generator, T: int, H: int, mode: str = "outlier",
                           lo: int = 8, hi: int = 12) -> np.ndarray:
    """bf16 bits [T][H] with a large dynamic range inside 32-element blocks (see the recipe above)."""
    x = rng.standard_normal((T, H), dtype=np.float32).reshape(T, H // 32, 32)
    if mode in ("outlier", "both"):
        pos = rng.integers(0, 32, size=(T, H // 32, 1))
        mul = np.exp2(rng.integers(lo, hi + 1, size=(T, H // 32, 1))).astype(np.float32)
        np.put_along_axis(x, pos, np.take_along_axis(x, pos, -1) * mul, -1)
    if mode in ("zeros", "both"):
        zero = rng.random((T, H // 32, 32)) < 0.5
        big = rng.random((T, H // 32, 1)) < 0.5
        x = np.where(zero, np.float32(0.0), np.where(big, x * np.float32(1024.0), x))
    if mode not in ("outlier", "zeros", "both"):
        raise ValueError(mode)
    return f32_to_bf16_bits(x.reshape(T, H))


def boost_gate_up_rows(rng: np.random.Generator, planes: dict, boost: int = 4) -> dict:
    """Copy of the planes with one gate row and the matching up row per 32 rows of
    every expert raised by `boost` in all their UE8M0 exponents (see the recipe above)."""
    out = {k: v.copy() for k, v in planes.items()}
    sc = out["w13_scales"]
    E, two_i, _ = sc.shape
    I = two_i // 2
    for e in range(E):
        rows = rng.integers(0, 32, size=I // 32) + 32 * np.arange(I // 32)
        sc[e, rows] += np.uint8(boost)
        sc[e, I + rows] += np.uint8(boost)
    return out


def routing_logits(rng: np.random.Generator, T: int, E: int, k: int):
    logits = rng.standard_normal((T, E), dtype=np.float32)
    ids = np.argsort(-logits, axis=1, kind="stable")[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, ids, axis=1)
    return ids, _softmax_rows(sel)


def zipf_popularity(rng: np.random.Generator, E: int, s: float = 1.1) -> np.ndarray:
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p_rank = ranks ** (-s)
    p_rank /= p_rank.sum()
    perm = rng.permutation(E)
    p = np.empty(E, dtype=np.float64)
    p[perm] = p_rank
    return p


def routing_zipf(rng: np.random.Generator, T: int, E: int, k: int, popularity=None):
    p = zipf_popularity(rng, E) if popularity is None else popularity
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        ids[t] = rng.choice(E, size=k, replace=False, p=p)
    weights = _softmax_rows(rng.standard_normal((T, k), dtype=np.float32))
    return ids, weights


def routing(rng: np.random.Generator, cfg: LayerConfig, T: int | None = None, popularity=None):
    T = cfg.tokens if T is None else T
    if cfg.routing == "logits":
        return routing_logits(rng, T, cfg.num_experts, cfg.top_k)
    return routing_zipf(rng, T, cfg.num_experts, cfg.top_k, popularity)


@dataclasses.dataclass
class LayerInputs:
    cfg: LayerConfig
    x: np.ndarray            # uint16 bf16 bits [T][H]
    ids: np.ndarray          # int32 [T][k]
    weights: np.ndarray      # float32 [T][k]
    planes: dict             # the four uint8 sections


def layer_inputs(cfg: LayerConfig, seed: int | None = None) -> LayerInputs:
    """Inputs of one configuration: planes first, then activations, then routing."""
    rng = rng_for(cfg.seed if seed is None else seed)
    planes = code_planes(rng, cfg.num_experts, cfg.hidden, cfg.inter, cfg.exp_lo, cfg.exp_hi)
    x = activations(rng, cfg.tokens, cfg.hidden)
    ids, weights = routing(rng, cfg)
    return LayerInputs(cfg, x, ids, weights, planes)


def small_layer_inputs(H: int, I: int, E: int, k: int, T: int, seed: int,
                       exp_lo: int = -9, exp_hi: int = -6, routing_kind: str = "logits") -> LayerInputs:
    cfg = LayerConfig(f"H{H}_I{I}_E{E}_k{k}_T{T}", H, I, E, k, T, exp_lo, exp_hi, routing_kind, seed)
    return layer_inputs(cfg)


@dataclasses.dataclass
class CachedLayerInputs:
    cfg: LayerConfig
    x: np.ndarray         # bf16 bits [T][H]
    ids: np.ndarray       # int32 [T][k] routed expert ids in [0, cfg.num_experts)
    weights: np.ndarray   # float32 [T][k]
    planes: dict          # planes of the S resident slots
    slot_of: np.ndarray   # int32 [cfg.num_experts]: slot of each routed expert, -1 if not resident


def cached_layer_inputs(cfg: LayerConfig, extra_slots: int = 0) -> CachedLayerInputs:
    """A layer of cfg.num_experts routed experts behind an expert cache: activations and
    routing first, then planes only for the step's routed experts plus `extra_slots`
    others, placed at slots in a random order."""
    rng = rng_for(cfg.seed)
    x = activations(rng, cfg.tokens, cfg.hidden)
    ids, weights = routing(rng, cfg)
    used = np.unique(ids)
    rest = np.setdiff1d(np.arange(cfg.num_experts), used)
    resident = np.concatenate([used, rng.choice(rest, size=min(extra_slots, len(rest)), replace=False)])
    slot_of = np.full(cfg.num_experts, -1, np.int32)
    slot_of[resident] = rng.permutation(len(resident)).astype(np.int32)
    planes = code_planes(rng, len(resident), cfg.hidden, cfg.inter, cfg.exp_lo, cfg.exp_hi)
    return CachedLayerInputs(cfg, x, ids, weights, planes, slot_of)


# --------------------------------------------------------------------------- NVFP4

def _e4m3_positive_table():
    """Values and bytes of the positive normal e4m3fn codes (exponent field 1..15)."""
    vals, codes = [], []
    for ef in range(1, 16):
        for m in range(8):
            if ef == 15 and m == 7:
                continue  # the NaN code
            vals.append((1.0 + m / 8.0) * 2.0 ** (ef - 7))
            codes.append((ef << 3) | m)
    return np.array(vals), np.array(codes, dtype=np.uint8)


def e4m3_round_positive(v: np.ndarray) -> np.ndarray:
    """Nearest positive normal e4m3fn byte to each value in [2^-6, 448) (ties: even mantissa)."""
    v = np.asarray(v, dtype=np.float64)
    f, e = np.frexp(v)                      # v = f * 2^e, f in [0.5, 1)
    m = np.rint((2.0 * f - 1.0) * 8.0)      # 3 mantissa bits of 1.m, ties to even
    carry = m == 8.0
    m = np.where(carry, 0.0, m).astype(np.int32)
    ef = (e - 1 + 7 + carry).astype(np.int32)   # biased exponent field
    return ((ef << 3) | m).astype(np.uint8)


@dataclasses.dataclass
class Nvfp4Tensors:
    e2m1: np.ndarray      # uint8 [n][rows][K/2], low nibble = even element
    e4m3: np.ndarray      # uint8 [n][rows][K/16]
    scale_2: np.ndarray   # float32 [n]


def nvfp4_tensors(rng: np.random.Generator, n: int, rows: int, K: int,
                  scale_2: float = 2.0 ** -8) -> Nvfp4Tensors:
    e2m1 = random_bytes(rng, (n, rows, K // 2))
    e = rng.uniform(-6.0, 2.0, size=(n, rows, K // 16))
    e4m3 = e4m3_round_positive(np.exp2(e))
    return Nvfp4Tensors(e2m1, e4m3, np.full(n, scale_2, dtype=np.float32))


def requant_inputs(cfg: RequantConfig = REQUANT, experts: int | None = None):
    """The re-quantizer workload: (gate/up tensors, down tensors).

    gate/up: 2*E tensors of [I][H] (expert e's gate is tensor 2e, its up tensor
    2e+1, so the outputs land contiguously in the w13 planes); down: E tensors of
    [H][I].  ``experts`` limits the draw to the first experts (same values as the
    full draw for those experts: every expert has its own child seed).
    """
    E = cfg.num_experts if experts is None else experts
    seeds = np.random.SeedSequence(cfg.seed).spawn(cfg.num_experts)
    gu_list, dn_list = [], []
    for e in range(E):
        rng = np.random.default_rng(seeds[e])
        gu_list.append(nvfp4_tensors(rng, 2, cfg.inter, cfg.hidden))
        dn_list.append(nvfp4_tensors(rng, 1, cfg.hidden, cfg.inter))
    gu = Nvfp4Tensors(np.concatenate([t.e2m1 for t in gu_list]),
                      np.concatenate([t.e4m3 for t in gu_list]),
                      np.concatenate([t.scale_2 for t in gu_list]))
    dn = Nvfp4Tensors(np.concatenate([t.e2m1 for t in dn_list]),
                      np.concatenate([t.e4m3 for t in dn_list]),
                      np.concatenate([t.scale_2 for t in dn_list]))
    return gu, dn


# --------------------------------------------------------------------------- FP8

@dataclasses.dataclass
class Fp8Tensors:
    w8: np.ndarray        # uint8 e4m3fn bytes [n][rows][K]
    scales: np.ndarray    # float32 [n][ceil(rows/128)][ceil(K/128)]


def fp8_tensors(rng: np.random.Generator, n: int, rows: int, K: int) -> Fp8Tensors:
    b = random_bytes(rng, (n, rows, K))
    nan = (b & 0x7F) == 0x7F
    b[nan] = rng.integers(0, 0x7F, size=int(nan.sum()), dtype=np.uint8) | (b[nan] & 0x80)   # no NaN codes
    sc = np.exp2(rng.uniform(-14.0, -8.0, size=(n, (rows + 127) // 128, (K + 127) // 128))).astype(np.float32)
    return Fp8Tensors(b, sc)


def requant_fp8_inputs(cfg: RequantConfig = REQUANT, experts: int = 16):
    """The FP8 loader workload: (gate/up tensors, down tensors) of the first `experts`
    experts, laid out as requant_inputs lays out the NVFP4 ones (a child seed each)."""
    seeds = np.random.SeedSequence(cfg.seed + 100).spawn(cfg.num_experts)
    gu, dn = [], []
    for e in range(experts):
        rng = np.random.default_rng(seeds[e])
        gu.append(fp8_tensors(rng, 2, cfg.inter, cfg.hidden))
        dn.append(fp8_tensors(rng, 1, cfg.hidden, cfg.inter))
    cat = lambda ts: Fp8Tensors(np.concatenate([t.w8 for t in ts]), np.concatenate([t.scales for t in ts]))
    return cat(gu), cat(dn)


# --------------------------------------------------------------------------- MXFP4

@dataclasses.dataclass
class Mxfp4Tensors:
    e2m1: np.ndarray      # uint8 [n][rows][K/2], low nibble = even element
    scales: np.ndarray    # uint8 UE8M0 bytes [n][rows][K/32]


def mxfp4_tensors(rng: np.random.Generator, n: int, rows: int, K: int, plus_zero_frac: float = 0.0) -> Mxfp4Tensors:
    """e2m1 nibbles uniform over all 16 values, scale exponents uniform in [-12, -2];
    with plus_zero_frac > 0 that fraction of the elements is replaced by +0
    (an export that writes every exact zero as +0)."""
    e2m1 = random_bytes(rng, (n, rows, K // 2))
    if plus_zero_frac > 0.0:
        nib = np.stack([e2m1 & 0xF, e2m1 >> 4], axis=-1)
        nib[rng.random(nib.shape) < plus_zero_frac] = 0
        nib[nib == 8] = 0
        e2m1 = (nib[..., 0] | (nib[..., 1] << 4)).astype(np.uint8)
    sc = (127 + rng.integers(-12, -1, size=(n, rows, K // 32))).astype(np.uint8)
    return Mxfp4Tensors(e2m1, sc)


def plus_zero_nvfp4(rng: np.random.Generator, n: int, rows: int, K: int, zero_frac: float = 0.25) -> Nvfp4Tensors:
    """NVFP4 tensors whose exact zeros are all +0 (nibble 0), about zero_frac of the elements."""
    t = nvfp4_tensors(rng, n, rows, K)
    nib = np.stack([t.e2m1 & 0xF, t.e2m1 >> 4], axis=-1)
    nib[rng.random(nib.shape) < zero_frac] = 0
    nib[nib == 8] = 0
    t.e2m1 = (nib[..., 0] | (nib[..., 1] << 4)).astype(np.uint8)
    return t


def requant_mxfp4_inputs(cfg: RequantConfig = REQUANT, experts: int = 16):
    """The MXFP4 loader workload: (gate/up tensors, down tensors) of the first `experts`
    experts, laid out as requant_inputs lays out the NVFP4 ones (a child seed each)."""
    seeds = np.random.SeedSequence(cfg.seed + 200).spawn(cfg.num_experts)
    gu, dn = [], []
    for e in range(experts):
        rng = np.random.default_rng(seeds[e])
        gu.append(mxfp4_tensors(rng, 2, cfg.inter, cfg.hidden))
        dn.append(mxfp4_tensors(rng, 1, cfg.hidden, cfg.inter))
    cat = lambda ts: Mxfp4Tensors(np.concatenate([t.e2m1 for t in ts]), np.concatenate([t.scales for t in ts]))
    return cat(gu), cat(dn)


# --------------------------------------------------------------------------- FP4 layer

def w4_planes(rng: np.random.Generator, E: int, H: int, I: int, scale_2: float = 2.0 ** -8) -> dict:
    """NVFP4 expert planes of the FP4 layer: e2m1 nibbles uniform over all 16 values,
    e4m3 block-16 scale bytes uniform over the positive codes of [2^-6, 4) (bytes 0x08 ..
    0x47: eight per binade, so the scales are close to log-uniform), one scale_2 per tensor
    (gate, up and down of every expert)."""
    def part(rows, K):
        e2m1 = random_bytes(rng, (E, rows, K // 2))
        e4m3 = rng.integers(0x08, 0x48, size=(E, rows, K // 16), dtype=np.uint8)
        return e2m1, e4m3
    w13_e2m1, w13_e4m3 = part(2 * I, H)
    w2_e2m1, w2_e4m3 = part(H, I)
    return {"w13_e2m1": w13_e2m1, "w13_e4m3": w13_e4m3,
            "w13_scale_2": np.full((E, 2), scale_2, np.float32),
            "w2_e2m1": w2_e2m1, "w2_e4m3": w2_e4m3,
            "w2_scale_2": np.full(E, scale_2, np.float32)}


@dataclasses.dataclass
class W4LayerInputs:
    cfg: LayerConfig
    x: np.ndarray
    ids: np.ndarray
    weights: np.ndarray
    planes: dict


def w4_layer_inputs(cfg: LayerConfig) -> W4LayerInputs:
    """Inputs of the FP4 layer for one configuration: planes, then activations, then routing."""
    rng = rng_for(cfg.seed)
    planes = w4_planes(rng, cfg.num_experts, cfg.hidden, cfg.inter)
    x = activations(rng, cfg.tokens, cfg.hidden)
    ids, weights = routing(rng, cfg)
    return W4LayerInputs(cfg, x, ids, weights, planes)
