"""Pins for the oracle's NVFP4 -> 2-bit re-quantizer (CPU only).

What fixes the result (page "The v0.24.0 port", section "Our hooks", modelopt.py
bullet; page "vLLM-Moet wiki", section "2-bit expert planes"): exact f64
dequantisation of e2m1 x e4m3 x scale_2; codes from {-4,-1,1,4}; one UE8M0
scale per block of 32 that absorbs scale_2; least squared error.  Pins:
  * brute force over all 252 UE8M0 exponents in exact rationals (tiny_exact),
    on random blocks shaped like the requant workload and on adversarial ones;
  * the per-element nearest code equals exhaustive search over code vectors;
  * exactly representable blocks come back with zero error, bit for bit;
  * negation flips only the code sign bits; a power-of-two scale_2 only moves u.
"""
import math
import random

import numpy as np
import pytest

import oracle
from oracle import tiny_exact
from bit_moe_expert_w2_gb300 import inputs


def _block_arrays(nibbles, e4m3_pair):
    """One block as (e2m1 [1][1][16], e4m3 [1][1][2]) arrays with K = 32."""
    b = np.zeros(16, np.uint8)
    for i, n in enumerate(nibbles):
        b[i // 2] |= (n & 15) << (4 * (i % 2))
    return b.reshape(1, 1, 16), np.array(e4m3_pair, np.uint8).reshape(1, 1, 2)


def _unpack_codes(code_bytes):
    return [(int(code_bytes[i // 4]) >> (2 * (i % 4))) & 3 for i in range(32)]


def _oracle_block(nibbles, e4m3_pair, scale_2):
    e2m1, e4m3 = _block_arrays(nibbles, e4m3_pair)
    codes, scales, st = oracle.requant(e2m1, e4m3, np.array([scale_2], np.float32))
    return _unpack_codes(codes.reshape(-1)), int(scales.reshape(-1)[0]), st


def _check_vs_bruteforce(nibbles, e4m3_pair, scale_2):
    codes, s, st = _oracle_block(nibbles, e4m3_pair, scale_2)
    ref = tiny_exact.requant_block(nibbles, e4m3_pair, float(np.float32(scale_2)))
    if ref is None:
        assert st == oracle.BAD_NVFP4 and s == 0 and codes == [0] * 32
    else:
        assert st == 0
        assert (codes, s) == (ref[0], ref[1]), (nibbles, e4m3_pair, scale_2)


def test_bruteforce_random_workload_blocks():
    t = inputs.nvfp4_tensors(np.random.default_rng(11), 1, 4, 32 * 10)
    blocks = 40
    for g in range(blocks):
        row, b = divmod(g, 10)
        byts = t.e2m1[0, row, b * 16:(b + 1) * 16]
        nib = [(int(byts[i // 2]) >> (4 * (i % 2))) & 15 for i in range(32)]
        sc = list(t.e4m3[0, row, 2 * b:2 * b + 2])
        _check_vs_bruteforce(nib, sc, float(t.scale_2[0]))


def test_bruteforce_random_any_e4m3_and_scale2():
    rnd = random.Random(3)
    for _ in range(40):
        nib = [rnd.randrange(16) for _ in range(32)]
        sc = [rnd.choice([b for b in range(256) if (b & 0x7F) != 0x7F]) for _ in range(2)]
        s2 = float(np.float32(rnd.uniform(0.5, 2) * 2.0 ** rnd.randint(-30, 30)))
        _check_vs_bruteforce(nib, sc, s2)


ADVERSARIAL = [
    # one large element and many tiny ones (widest spread of magnitudes in a block)
    ([0b0111] + [0b0001] * 31, [0x7E, 0x01], 1.0),
    ([0b0111] + [0b0001] * 15 + [0] * 16, [0x7E, 0x01], 1.0),
    # all zeros (+0 and -0): smallest scale, codes by sign bit
    ([0] * 16 + [8] * 16, [0x38, 0x38], 1.0),
    ([8] * 32, [0x38, 0xB8], 2.0 ** -8),
    # negative e4m3 scale: signs flip with it
    ([0b0011, 0b1011] * 16, [0xB8, 0x38], 1.0),
    # exact code ties: |x| = 2.5 * 2^u for some u in range
    ([0b0101, 0b0100, 0b0010, 0b0001] * 8, [0x3A, 0x38], 1.0),
    # equal elements of magnitude 1*2^u: SSE 0 at u and at u-2 (tie -> smaller u)
    ([0b0010] * 32, [0x38, 0x38], 1.0),
    ([0b0110] * 32, [0x38, 0x38], 2.0 ** -8),
    # subnormal e4m3, tiny scale_2 (near the bottom clamp u = -126)
    ([0b0111, 0b0001] * 16, [0x01, 0x07], 2.0 ** -126),
    ([0b0111] * 32, [0x01, 0x01], float(np.float32(2.0 ** -149))),
    ([0b0001] * 32, [0x01, 0x01], float(np.float32(2.0 ** -140))),
    # huge scale_2 (top clamp u = 125)
    ([0b0111] * 32, [0x7E, 0x7E], float(np.float32(2.0 ** 127))),
    ([0b0001, 0b0111] * 16, [0x08, 0x7E], float(np.float32(3.0e38))),
    # invalid inputs
    ([1] * 32, [0x7F, 0x38], 1.0),
    ([1] * 32, [0x38, 0xFF], 1.0),
    ([1] * 32, [0x38, 0x38], 0.0),
    ([1] * 32, [0x38, 0x38], -1.0),
    ([1] * 32, [0x38, 0x38], float("inf")),
    ([1] * 32, [0x38, 0x38], float("nan")),
]


@pytest.mark.parametrize("case", range(len(ADVERSARIAL)))
def test_bruteforce_adversarial(case):
    _check_vs_bruteforce(*ADVERSARIAL[case])


def test_nearest_code_equals_exhaustive_search():
    from fractions import Fraction
    rnd = random.Random(5)
    for n in (2, 3, 4, 5):
        for _ in range(6):
            u = rnd.randint(-3, 3)
            vals = [Fraction(rnd.choice([-1, 1]) * rnd.randint(0, 48), 8) * Fraction(2) ** u for _ in range(n)]
            # include an exact tie at 2.5*2^u now and then
            if rnd.random() < 0.5:
                vals[0] = Fraction(5, 2) * Fraction(2) ** u
            codes, _ = tiny_exact.nearest_codes_by_enumeration(vals, u)
            step = Fraction(2) ** u
            mine = [(1 if v < 0 else 0) << 1 | (1 if abs(v) > Fraction(5, 2) * step else 0) for v in vals]
            for c, m, v in zip(codes, mine, vals):
                if v == 0:
                    assert (c & 1) == 0
                else:
                    assert c == m


def _nvfp4_encode_codebook_block(rnd, u, k):
    """A block whose values are exactly +-{1,4} * 2^u, written as NVFP4 with scale_2 = 2^k."""
    codes = [rnd.randrange(4) for _ in range(32)]
    nib = [(8 if c & 2 else 0) | (0b0110 if c & 1 else 0b0010) for c in codes]
    e = u - k                      # e4m3 value 2^e (normal: exponent field e+7 in [1,15])
    byte = (e + 7) << 3
    return codes, nib, [byte, byte], float(2.0 ** k)


def test_exactly_representable_blocks_roundtrip():
    rnd = random.Random(9)
    for _ in range(200):
        k = rnd.randint(-20, 20)
        u = k + rnd.randint(-6, 7)
        codes, nib, sc, s2 = _nvfp4_encode_codebook_block(rnd, u, k)
        got, s, st = _oracle_block(nib, sc, s2)
        assert st == 0
        x = [oracle.code_value(c) * 2.0 ** u for c in codes]
        y = [oracle.code_value(c) * 2.0 ** (s - 127) for c in got]
        assert x == y
        if any(c & 1 for c in codes):
            assert got == codes and s == u + 127
        else:  # all magnitude 1: the same values at u-2 with magnitude 4 (smaller u wins)
            assert s == u + 125 and got == [c | 1 for c in codes]


def test_negation_flips_only_code_signs():
    t = inputs.nvfp4_tensors(np.random.default_rng(21), 2, 8, 256)
    neg = inputs.Nvfp4Tensors(t.e2m1 ^ np.uint8(0x88), t.e4m3, t.scale_2)
    c1, s1, _ = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    c2, s2, _ = oracle.requant(neg.e2m1, neg.e4m3, neg.scale_2)
    assert np.array_equal(s1, s2)
    assert np.array_equal(c1 ^ np.uint8(0xAA), c2)


def test_power_of_two_scale2_moves_only_the_exponent():
    t = inputs.nvfp4_tensors(np.random.default_rng(22), 1, 8, 256)
    c1, s1, _ = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    c2, s2, _ = oracle.requant(t.e2m1, t.e4m3, t.scale_2 * np.float32(2.0 ** 5))
    assert np.array_equal(c1, c2)
    assert np.array_equal(s1.astype(int) + 5, s2.astype(int))


def test_f64_sse_agrees_for_power_of_two_scale2():
    # With scale_2 a power of two every value has at most 6 significant bits, so
    # the plain f64 squared error is exact for every scale near the data (the far
    # ones are larger by many orders of magnitude): an independent numpy argmin
    # over all 252 exponents must agree with the oracle.
    t = inputs.nvfp4_tensors(np.random.default_rng(23), 1, 16, 256)
    codes, scales, _ = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    e2m1_mag = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    byts = t.e2m1.reshape(-1)
    nib = np.stack([byts & 15, byts >> 4], axis=1).reshape(-1)
    sign = np.where(nib & 8, -1.0, 1.0)
    mag = e2m1_mag[nib & 7]
    e4 = np.array([oracle.e4m3_value(int(b)) for b in t.e4m3.reshape(-1)])
    x = (sign * mag * np.repeat(e4, 16) * float(t.scale_2[0])).reshape(-1, 32)
    a = np.abs(x)
    us = np.arange(-126, 126)
    step = np.exp2(us.astype(np.float64))[:, None, None]
    v = np.where(a[None] > 2.5 * step, 4 * step, step)
    sse = ((a[None] - v) ** 2).sum(axis=2)          # [u][block]
    best = us[np.argmin(sse, axis=0)]                # first minimum = smaller u on ties
    assert np.array_equal(best + 127, scales.reshape(-1).astype(int))


def test_sampled_blocks_match_whole_tensor_path():
    t = inputs.nvfp4_tensors(np.random.default_rng(24), 3, 4, 128)
    codes, scales, st = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    ids = np.array([0, 5, 17, 31, 47], np.int64)
    c2, s2, st2 = oracle.requant_blocks(t.e2m1, t.e4m3, t.scale_2, ids)
    assert np.array_equal(c2, codes.reshape(-1, 8)[ids])
    assert np.array_equal(s2, scales.reshape(-1)[ids])
