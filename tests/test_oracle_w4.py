"""Pins for the oracle's FP4 layer (CPU only).

What fixes the result: page "vLLM-Moet wiki", sections "The kernels" and "FP4
recovery" (moe_w4_mm: the same MoE forward over the NVFP4 experts, twice the
plane bytes); page "The v0.24.0 port", "Our hooks", modelopt.py bullet (NVFP4 =
e2m1 x e4m3 block-16 x per-tensor scale_2, exact in f64).  Pins, each from an
independent route:
  * NVFP4 experts whose values are exactly 2-bit planes values (e2m1 in {+-1,
    +-4}, one power-of-two e4m3 scale per 32 elements, power-of-two scale_2)
    give, through the FP4 layer, y and h bitwise equal to the 2-bit layer over
    the planes the NVFP4 re-quantizer writes for them;
  * one expert, top-1, weight 1 equals a dense SwiGLU MLP in torch f64 from
    weights decoded here by exact rationals (tiny_exact's e2m1 / e4m3 tables);
  * each tensor's scale_2 acts on its own projection: doubling down's doubles y
    exactly, doubling gate's and up's changes h as the dense model says;
  * an e4m3 NaN scale zeroes its 16 weights and sets status bit 2;
  * the OpenMP build agrees bitwise.
"""
import numpy as np
import torch

import oracle
from oracle import tiny_exact
from bit_moe_expert_w2_gb300 import inputs

BAD_SCALE = 2


def _decode_w4(e2m1, e4m3, s2):
    """Dense f64 weights [rows][K] of one NVFP4 tensor, from exact rationals."""
    rows, half_k = e2m1.shape
    K = 2 * half_k
    nib_val = np.array([(-1.0 if n else 1.0) * float(m) for n, m in (tiny_exact.e2m1(i) for i in range(16))])
    sc_val = np.array([np.nan if v is None else (-1.0 if v[0] else 1.0) * float(v[1])
                       for v in (tiny_exact.e4m3(b) for b in range(256))])
    nib = np.stack([e2m1 & 0xF, e2m1 >> 4], axis=-1).reshape(rows, K)
    return nib_val[nib] * np.repeat(sc_val[e4m3], 16, axis=-1) * float(s2)


def _bf16_round(a):
    a = np.asarray(a, dtype=np.float64)
    f, e = np.frexp(a)
    return np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)


def _representable_planes(rng, E, H, I):
    """NVFP4 planes whose every 32-element block is exactly +-{1,4} x 2^u."""
    def part(rows, K):
        nib = rng.choice(np.array([2, 6, 10, 14], np.uint8), size=(E, rows, K))
        e2m1 = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        k32 = rng.integers(-4, 3, size=(E, rows, K // 32))          # e4m3 = 2^k, one per 32
        e4m3 = np.repeat(((k32 + 7) << 3).astype(np.uint8), 2, axis=-1)
        return e2m1, e4m3
    a, b = part(2 * I, H)
    c, d = part(H, I)
    s13 = np.exp2(rng.integers(-9, -6, size=(E, 2))).astype(np.float32)
    s2 = np.exp2(rng.integers(-9, -6, size=E)).astype(np.float32)
    return {"w13_e2m1": a, "w13_e4m3": b, "w13_scale_2": s13, "w2_e2m1": c, "w2_e4m3": d, "w2_scale_2": s2}


def test_representable_experts_match_the_2bit_layer_over_requant_planes():
    rng = np.random.default_rng(1)
    E, H, I, T, k = 3, 128, 96, 4, 2
    p4 = _representable_planes(rng, E, H, I)
    # gate and up re-quantized as separate tensors (their own scale_2), down as one
    gate = oracle.requant(p4["w13_e2m1"][:, :I], p4["w13_e4m3"][:, :I], p4["w13_scale_2"][:, 0])
    up = oracle.requant(p4["w13_e2m1"][:, I:], p4["w13_e4m3"][:, I:], p4["w13_scale_2"][:, 1])
    dn = oracle.requant(p4["w2_e2m1"], p4["w2_e4m3"], p4["w2_scale_2"])
    assert gate[2] == up[2] == dn[2] == 0
    p2 = {"w13_codes": np.concatenate([gate[0], up[0]], axis=1), "w13_scales": np.concatenate([gate[1], up[1]], axis=1),
          "w2_codes": dn[0], "w2_scales": dn[1]}
    x = inputs.activations(rng, T, H)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    y4, h4, st4 = oracle.forward_tokens_w4(x, ids, w, p4, want_h=True)
    y2, h2, st2 = oracle.forward_tokens(x, ids, w, p2, want_h=True)
    assert st4 == st2 == 0
    assert np.array_equal(h4, h2) and np.array_equal(y4, y2)


def test_one_expert_top1_equals_dense_swiglu():
    rng = np.random.default_rng(2)
    H, I, T = 128, 64, 5
    p = inputs.w4_planes(rng, 1, H, I, scale_2=2.0 ** -4)
    p["w13_scale_2"][0] = [2.0 ** -4, 2.0 ** -3]
    p["w2_scale_2"][0] = 2.0 ** -5
    x = inputs.activations(rng, T, H)
    y, st = oracle.forward_tokens_w4(x, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), p)
    Wg = torch.from_numpy(_decode_w4(p["w13_e2m1"][0, :I], p["w13_e4m3"][0, :I], p["w13_scale_2"][0, 0]))
    Wu = torch.from_numpy(_decode_w4(p["w13_e2m1"][0, I:], p["w13_e4m3"][0, I:], p["w13_scale_2"][0, 1]))
    W2 = torch.from_numpy(_decode_w4(p["w2_e2m1"][0], p["w2_e4m3"][0], p["w2_scale_2"][0]))
    xt = torch.from_numpy(oracle.bf16_bits_to_f64(x))
    h = torch.from_numpy(_bf16_round((torch.nn.functional.silu(xt @ Wg.T) * (xt @ Wu.T)).numpy()))
    ref = _bf16_round((h @ W2.T).numpy())
    assert st == 0
    assert np.array_equal(oracle.bf16_bits_to_f64(y), ref)


def test_each_scale_2_acts_on_its_own_projection():
    rng = np.random.default_rng(3)
    lay = inputs.w4_layer_inputs(inputs.LayerConfig("w4s", 128, 64, 4, 2, 3, -9, -6, "logits", 4))
    y0, h0, _ = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes, want_h=True)
    p = {n: v.copy() for n, v in lay.planes.items()}
    p["w2_scale_2"] *= 2
    y1, h1, _ = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, p, want_h=True)
    assert np.array_equal(h0, h1)
    f0, f1 = oracle.bf16_bits_to_f64(y0), oracle.bf16_bits_to_f64(y1)
    assert np.array_equal(f1, 2 * f0)
    # gate's scale_2 halves g (h changes), up's doubling doubles u: h = bf16(SiLU(g) u)
    q = {n: v.copy() for n, v in lay.planes.items()}
    q["w13_scale_2"][:, 1] *= 2
    _, h2, _ = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, q, want_h=True)
    assert np.array_equal(oracle.bf16_bits_to_f64(h2), 2 * oracle.bf16_bits_to_f64(h0))


def test_nan_scale_zeroes_its_16_weights():
    rng = np.random.default_rng(5)
    lay = inputs.w4_layer_inputs(inputs.LayerConfig("w4n", 64, 64, 2, 1, 2, -9, -6, "logits", 6))
    p = {n: v.copy() for n, v in lay.planes.items()}
    e = int(lay.ids[0, 0])
    p["w2_e4m3"][e, 5, 1] = 0x7F                      # NaN: down row 5, elements 16..31
    z = {n: v.copy() for n, v in lay.planes.items()}
    nib = z["w2_e2m1"][e, 5]
    nib[8:16] = 0                                      # the same 16 weights as +0
    y1, st1 = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, p)
    y0, st0 = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, z)
    assert st1 == BAD_SCALE and st0 == 0
    assert np.array_equal(y0, y1)


def test_parallel_build_agrees():
    lay = inputs.w4_layer_inputs(inputs.LayerConfig("w4p", 128, 64, 6, 3, 9, -9, -6, "logits", 7))
    a = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes)
    b = oracle.forward_tokens_w4(lay.x, lay.ids, lay.weights, lay.planes, parallel=True)
    assert np.array_equal(a[0], b[0]) and a[1] == b[1]
