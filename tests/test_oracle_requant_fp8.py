"""Pins for the oracle's FP8 block-128 -> 2-bit re-quantizer (CPU only).

What fixes the result (page "The v0.24.0 port", section "Our hooks", fp8.py
bullet: the FP8 block-quant loader re-quantizes fp8 weights with f32 block-128
scales to the sign-symmetric codebook in float64; page "vLLM-Moet wiki",
section "2-bit expert planes"): each element is e4m3 x the f32 scale of its
128 x 128 block, exactly; then, as for NVFP4, one UE8M0 scale per 32 elements
and codes from {-4,-1,1,4} at least squared error.  Pins:
  * brute force over all 252 UE8M0 exponents in exact rationals (tiny_exact),
    on workload-shaped, random and adversarial blocks;
  * the same real numbers give the same codes and scale byte through the NVFP4
    loader (e2m1 values are e4m3 values; a power-of-two scale_2 folds into S);
  * each 32-element block takes the scale of its own 128 x 128 block (power-of-
    two scales per block only move the UE8M0 byte);
  * exactly representable blocks come back with zero error, bit for bit;
  * the OpenMP build agrees bitwise.
"""
import random
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny_exact
from bit_moe_expert_w2_gb300 import inputs

CODE = [1, 4, -1, -4]


def _codes(code_bytes):
    return [(int(code_bytes[i // 4]) >> (2 * (i % 4))) & 3 for i in range(32)]


def _oracle_block(byts, scale):
    w8 = np.array(byts, np.uint8).reshape(1, 1, 32)
    c, u, st = oracle.requant_fp8(w8, np.array([[[scale]]], np.float32))
    return _codes(c.reshape(-1)), int(u.reshape(-1)[0]), st


def _check(byts, scale):
    codes, s, st = _oracle_block(byts, scale)
    ref = tiny_exact.requant_block_fp8(byts, float(np.float32(scale)))
    if ref is None:
        assert st == oracle.BAD_NVFP4 and s == 0 and codes == [0] * 32
    else:
        assert st == 0 and (codes, s) == (ref[0], ref[1]), (byts, scale)


NON_NAN = [b for b in range(256) if (b & 0x7F) != 0x7F]


def test_bruteforce_workload_blocks():
    t = inputs.fp8_tensors(np.random.default_rng(21), 1, 4, 256)
    for r in range(4):
        for b in range(8):
            _check(list(t.w8[0, r, 32 * b:32 * b + 32]), float(t.scales[0, 0, (32 * b) // 128]))


def test_bruteforce_random_bytes_and_scales():
    rnd = random.Random(5)
    for _ in range(40):
        byts = [rnd.choice(NON_NAN) for _ in range(32)]
        s = float(np.float32(rnd.uniform(0.5, 2.0) * 2.0 ** rnd.randint(-40, 40)))
        _check(byts, s)


ADVERSARIAL = [
    ([0x7E] + [0x01] * 31, 1.0),                       # 448 beside the smallest subnormal
    ([0x7E] + [0x00] * 31, 2.0 ** -100),                # one element, the rest +0
    ([0x00] * 16 + [0x80] * 16, 1.0),                   # all zeros: smallest scale, codes by sign
    ([0x80] * 32, 3.0),                                 # all -0
    ([0x38, 0xB8] * 16, 2.0 ** -126),                   # +-1 at the bottom of the f32 range
    ([0x7E] * 32, float(np.float32(3.0e38))),           # near the top of the UE8M0 range
    ([0x01, 0x02, 0x03, 0x04] * 8, float(np.float32(1e-38))),   # subnormal scale
    ([0x3C] * 32, 1.0),                                 # 1.5: between codes 1 and 4 at u = -1 / 0
    ([0x45] * 32, 1.0),                                 # 2.5: the exact code tie at u = 0
    ([0x38] * 31 + [0x7F], 1.0),                        # an e4m3 NaN: invalid block
    ([0x38] * 32, 0.0),                                 # zero scale: invalid
    ([0x38] * 32, -1.0),                                # negative scale: invalid
    ([0x38] * 32, float("inf")),                        # infinite scale: invalid
    ([0x38] * 32, float("nan")),                        # NaN scale: invalid
]


@pytest.mark.parametrize("byts,scale", ADVERSARIAL)
def test_bruteforce_adversarial_blocks(byts, scale):
    _check(byts, scale)


def test_same_values_through_the_nvfp4_loader_give_the_same_planes():
    # e2m1 values are e4m3 values: nibble n -> e4m3 byte of the same value; with
    # equal e4m3 block scales and a power-of-two scale_2 the f32 FP8 scale
    # S = e4m3(s) * scale_2 is exact, so both loaders see the same 32 numbers
    e2m1_to_e4m3 = {}
    for nib in range(16):
        neg, mag = tiny_exact.e2m1(nib)
        for b in range(256):
            v = tiny_exact.e4m3(b)
            if v is not None and v == (neg, mag) and (mag != 0 or ((b >> 7) & 1) == neg):
                e2m1_to_e4m3[nib] = b
                break
    assert len(e2m1_to_e4m3) == 16
    rng = np.random.default_rng(8)
    for _ in range(30):
        nib = rng.integers(0, 16, 32)
        sbyte = int(rng.choice([b for b in NON_NAN if b < 0x80 and b > 0]))
        s2 = np.float32(2.0 ** int(rng.integers(-20, 5)))
        e2m1 = np.zeros(16, np.uint8)
        for i, n in enumerate(nib):
            e2m1[i // 2] |= int(n) << (4 * (i % 2))
        c1, u1, st1 = oracle.requant(e2m1.reshape(1, 1, 16), np.array([sbyte, sbyte], np.uint8).reshape(1, 1, 2),
                                     np.array([s2], np.float32))
        S = np.float32(float(tiny_exact.e4m3(sbyte)[1] * Fraction(float(s2))))
        assert Fraction(float(S)) == tiny_exact.e4m3(sbyte)[1] * Fraction(float(s2))
        w8 = np.array([e2m1_to_e4m3[int(n)] for n in nib], np.uint8).reshape(1, 1, 32)
        c2, u2, st2 = oracle.requant_fp8(w8, np.array([[[S]]], np.float32))
        assert st1 == st2 == 0 and np.array_equal(c1, c2) and np.array_equal(u1, u2)


def test_each_block_takes_the_scale_of_its_128x128_tile():
    # one 128 x 128 pattern repeated over 2 x 3 tiles (rows 256, K 384, plus a
    # ragged last row block of 16 rows), a power-of-two scale per tile: the
    # codes repeat and each block's UE8M0 byte moves by its tile's exponent
    base = inputs.fp8_tensors(np.random.default_rng(9), 1, 128, 128).w8[0]
    rows, K = 272, 384
    w8 = np.tile(base, (3, 3))[:rows, :K].reshape(1, rows, K)
    exps = np.array([[0, 3, -5], [7, -2, 1], [4, 0, -9]])
    sc = np.exp2(exps).astype(np.float32).reshape(1, 3, 3)
    c, u, st = oracle.requant_fp8(np.ascontiguousarray(w8), sc)
    c0, u0, _ = oracle.requant_fp8(np.ascontiguousarray(base.reshape(1, 128, 128)), np.ones((1, 1, 1), np.float32))
    assert st == 0
    for r in range(rows):
        for b in range(K // 32):
            tr, tc = r // 128, (32 * b) // 128
            assert np.array_equal(c[0, r, 8 * b:8 * b + 8], c0[0, r % 128, 8 * (b % 4):8 * (b % 4) + 8])
            want = int(u0[0, r % 128, b % 4]) + int(exps[tr, tc])
            assert int(u[0, r, b]) == want


def test_exactly_representable_blocks_round_trip():
    rng = np.random.default_rng(10)
    for _ in range(50):
        codes = rng.integers(0, 4, 32)
        u = int(rng.integers(-60, 60))
        byts = [{0: 0x38, 1: 0x48, 2: 0xB8, 3: 0xC8}[int(c)] for c in codes]   # +1, +4, -1, -4
        c2, s, st = _oracle_block(byts, float(2.0 ** u))
        assert st == 0
        back = [CODE[c] * 2.0 ** (s - 127) for c in c2]
        assert back == [CODE[int(c)] * 2.0 ** u for c in codes]


def test_parallel_build_agrees():
    t = inputs.fp8_tensors(np.random.default_rng(12), 3, 200, 512)
    t.w8[1, 5, 40] = 0x7F
    t.scales[2, 0, 1] = 0.0
    a = oracle.requant_fp8(t.w8, t.scales)
    b = oracle.requant_fp8(t.w8, t.scales, parallel=True)
    assert all(np.array_equal(x, y) for x, y in zip(a[:2], b[:2])) and a[2] == b[2] == oracle.BAD_NVFP4
