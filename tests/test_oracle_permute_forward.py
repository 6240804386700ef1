"""Pins for the oracle's routing permutation and expert forward (CPU only).

Permutation (page "The v0.24.0 port", section "Our hooks", "Deterministic
unpermute" bullet): valid sorted ids are a permutation of token*top_k+j grouped
by expert; pinned to numpy's stable argsort and to the identity of
gather-then-unpermute.

Forward (page "vLLM-Moet wiki", sections "2-bit expert planes" and "The
kernels"; the SwiGLU expert MLP with SiLU(gate)*up between the grouped GEMMs):
pinned by closed forms on constant planes, by the one-expert top-1 special case
that must equal a dense SwiGLU MLP computed with torch in f64 from weights
decoded here independently, and by linearity in the router weights.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_moe_expert_w2_gb300 import inputs


# ----------------------------------------------------------------- permutation

@pytest.mark.parametrize("T,k,E,seed", [(4, 2, 8, 0), (1, 8, 256, 1), (32, 8, 256, 2),
                                        (257, 3, 17, 3), (0, 4, 8, 4), (50, 16, 5, 5)])
def test_permute_equals_stable_argsort(T, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    sorted_pairs, inv, offsets, st = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    ref = np.argsort(flat, kind="stable")
    assert np.array_equal(sorted_pairs, ref.astype(np.int32))
    assert np.array_equal(inv[sorted_pairs], np.arange(T * k))
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    assert st == 0


def test_permute_invalid_ids_go_last_and_flag():
    ids = np.array([[3, -1], [9, 0], [3, 100], [2, 3]], np.int32)
    sorted_pairs, inv, offsets, st = oracle.permute(ids, 8)
    key = np.where((ids >= 0) & (ids < 8), ids, 8).reshape(-1)
    assert np.array_equal(sorted_pairs, np.argsort(key, kind="stable"))
    assert offsets[-1] == 5 and st == oracle.BAD_EXPERT_ID


def test_gather_then_unpermute_is_identity():
    rng = np.random.default_rng(3)
    T, k, E, H = 37, 4, 11, 16
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    x = rng.standard_normal((T, H))
    sorted_pairs, inv, _, _ = oracle.permute(ids, E)
    x_perm = x[sorted_pairs // k]                    # rows grouped by expert
    back = x_perm[inv].reshape(T, k, H)              # slot t*k+j
    for j in range(k):
        assert np.array_equal(back[:, j], x)


# ----------------------------------------------------------------- forward

CODE_VALUES = np.array([1.0, 4.0, -1.0, -4.0])       # reading R1 (sign-magnitude)


def _decode_planes(codes, scales):
    """Dense f64 weights from codes [..., K/4] and UE8M0 bytes [..., K/32]."""
    shifts = np.array([0, 2, 4, 6], np.uint8)
    c = (codes[..., None] >> shifts) & 3
    c = c.reshape(*codes.shape[:-1], codes.shape[-1] * 4)
    s = np.repeat(np.exp2(scales.astype(np.float64) - 127.0), 32, axis=-1)
    return CODE_VALUES[c] * s


def _bf16_round(a):
    a = np.asarray(a, dtype=np.float64)
    f, e = np.frexp(a)
    return np.ldexp(np.rint(np.ldexp(f, 8)), e - 8)   # 8 significant bits, ties to even (normal range)


def _bf16_bits(v):
    return (np.asarray(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _constant_planes(E, H, I, gate_code, gate_s, up_code, up_s, down_code, down_s):
    byte = lambda c: np.uint8(c | (c << 2) | (c << 4) | (c << 6))
    w13c = np.empty((E, 2 * I, H // 4), np.uint8)
    w13c[:, :I] = byte(gate_code)
    w13c[:, I:] = byte(up_code)
    w13s = np.empty((E, 2 * I, H // 32), np.uint8)
    w13s[:, :I] = gate_s
    w13s[:, I:] = up_s
    return {"w13_codes": w13c, "w13_scales": w13s,
            "w2_codes": np.full((E, H, I // 4), byte(down_code), np.uint8),
            "w2_scales": np.full((E, H, I // 32), down_s, np.uint8)}


def test_closed_form_all_plus_one():
    H = I = 32
    planes = _constant_planes(2, H, I, 0, 127, 0, 127, 0, 127)
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x3F80                                  # 1.0
    ids = np.array([[1]], np.int32)
    w = np.array([[1.0]], np.float32)
    y, h, st = oracle.forward_tokens(x, ids, w, planes, want_h=True)
    # g = u = 1; h = bf16(SiLU(1)) = bf16(0.7310585786...) = 0.73046875; y = 32*h
    assert np.all(oracle.bf16_bits_to_f64(h) == 0.73046875)
    assert np.all(oracle.bf16_bits_to_f64(y) == 23.375) and st == 0


def test_closed_form_signs_scales_and_weights():
    H = I = 32
    # gate +4 * 2^-3, up -1 * 2^0, down +1 * 2^-5
    planes = _constant_planes(3, H, I, 1, 124, 2, 127, 0, 122)
    x = np.zeros((1, H), np.uint16)
    x[0, 5] = 0x4000                                  # 2.0
    ids = np.array([[2, 0]], np.int32)
    w = np.array([[0.5, 0.0]], np.float32)
    y, st = oracle.forward_tokens(x, ids, w, planes)
    # g = 1, u = -2 -> h = bf16(-2*SiLU(1)) = -1.4609375; d = 32 * h / 32; y = 0.5 * d
    assert np.all(oracle.bf16_bits_to_f64(y) == -0.73046875) and st == 0


def test_one_expert_top1_equals_dense_swiglu():
    lay = inputs.small_layer_inputs(H=128, I=96, E=1, k=1, T=5, seed=12, exp_lo=-4, exp_hi=-1)
    w = np.ones((5, 1), np.float32)
    ids = np.zeros((5, 1), np.int32)
    y, st = oracle.forward_tokens(lay.x, ids, w, lay.planes)
    W13 = torch.from_numpy(_decode_planes(lay.planes["w13_codes"][0], lay.planes["w13_scales"][0]))
    W2 = torch.from_numpy(_decode_planes(lay.planes["w2_codes"][0], lay.planes["w2_scales"][0]))
    x = torch.from_numpy(oracle.bf16_bits_to_f64(lay.x))
    I = 96
    g, u = x @ W13[:I].T, x @ W13[I:].T
    h = torch.from_numpy(_bf16_round((torch.nn.functional.silu(g) * u).numpy()))
    ref = _bf16_round((h @ W2.T).numpy())
    assert st == 0
    assert np.array_equal(oracle.bf16_bits_to_f64(y), ref)


def test_linearity_duplicates_and_zero_weight():
    lay = inputs.small_layer_inputs(H=64, I=64, E=4, k=2, T=3, seed=13)
    # one token routed twice to expert 2 with weights a and b equals once with a+b
    x = lay.x[:1]
    y_dup, _ = oracle.forward_tokens(x, np.array([[2, 2]], np.int32), np.array([[0.25, 0.5]], np.float32), lay.planes)
    y_one, _ = oracle.forward_tokens(x, np.array([[2, 1]], np.int32), np.array([[0.75, 0.0]], np.float32), lay.planes)
    assert np.array_equal(y_dup, y_one)
    # an invalid id contributes nothing and is flagged
    y_bad, st = oracle.forward_tokens(x, np.array([[2, 99]], np.int32), np.array([[0.75, 0.3]], np.float32), lay.planes)
    assert np.array_equal(y_bad, y_one) and st == oracle.BAD_EXPERT_ID


def test_bad_scale_byte_zeroes_its_block():
    lay = inputs.small_layer_inputs(H=64, I=64, E=2, k=1, T=1, seed=14)
    planes = {k: v.copy() for k, v in lay.planes.items()}
    planes["w2_scales"][1, :, :] = 0                  # every block of expert 1's down rows
    y, st = oracle.forward_tokens(lay.x, np.array([[1]], np.int32), np.array([[1.0]], np.float32), planes)
    assert np.all(oracle.bf16_bits_to_f64(y) == 0.0) and st == oracle.BAD_SCALE


@pytest.mark.parametrize("s", [0, 1, 126, 252, 253, 254, 255])
def test_ue8m0_validity_range_of_down_blocks(s):
    # Bytes 1..252 scale by 2^(s-127); 0 and 253..255 are outside the accepted
    # range (4 * 2^(s-127) must stay a normal bf16/fp32) and zero their block with
    # status bit 2.  Near the top g = u = 2^-8 gives a small h, so 2^125 times it
    # stays finite; near the bottom g = u = 1 keeps 2^-126 times it normal.
    H = I = 32
    planes = _constant_planes(1, H, I, 0, 127, 0, 127, 0, s)
    g = u = 1.0 if s < 128 else 2.0 ** -8
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = _bf16_bits(g)[()]
    y, st = oracle.forward_tokens(x, np.array([[0]], np.int32), np.array([[1.0]], np.float32), planes)
    h = _bf16_round(g / (1.0 + np.exp(-g)) * u)
    valid = 1 <= s <= 252
    want = _bf16_round(32.0 * h * 2.0 ** (s - 127)) if valid else 0.0
    got = oracle.bf16_bits_to_f64(y)
    assert np.all(np.isfinite(got)) and np.all(got == want)
    assert st == (0 if valid else oracle.BAD_SCALE)


@pytest.mark.parametrize("s", [252, 253])
def test_ue8m0_validity_range_of_gate_up_blocks(s):
    # x = 2^-128 (a bf16 subnormal); at s = 252 g = u = 2^125 * 2^-128 = 1/8, at
    # s = 253 the gate and up blocks count as zero, so h = 0 and y = 0.
    H = I = 32
    planes = _constant_planes(1, H, I, 0, s, 0, s, 0, 127)
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = 0x0020                                  # 32 * 2^-133 = 2^-128
    assert oracle.bf16_bits_to_f64(x)[0, 0] == 2.0 ** -128
    y, st = oracle.forward_tokens(x, np.array([[0]], np.int32), np.array([[1.0]], np.float32), planes)
    g = u = 0.125
    want = _bf16_round(32.0 * _bf16_round(g / (1.0 + np.exp(-g)) * u)) if s == 252 else 0.0
    assert np.all(oracle.bf16_bits_to_f64(y) == want)
    assert st == (0 if s == 252 else oracle.BAD_SCALE)
