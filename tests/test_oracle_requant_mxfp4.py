"""Pins for the oracle's MXFP4 loader and the zero-sign balancing option (CPU only).

What fixes the result: page "The v0.24.0 port", section "Our hooks", mxfp4.py
bullet (the FP4-checkpoint path builds the 2-bit planes at load) and page
"vLLM-Moet wiki" (FP4 experts load by a codes remap); an MXFP4 element is
e2m1 x 2^(s-127) with one UE8M0 byte s per 32 elements, and the planes follow
the same least-squares rule as the other loaders.  Zero-sign balancing: page
"vLLM-Moet wiki", the Kimi-K2.7 paragraph (an export writing every exact zero
as +0 biases the codes); with the option the exact zeros of a block take the
signs +,-,+,- in element order.  Pins:
  * brute force over all 252 UE8M0 exponents in exact rationals (tiny_exact), on
    random blocks at every kind of scale byte (middle, 0, 1, 253, 254);
  * the codes remap: away from the ends of the exponent range, the codes do not
    depend on the scale byte and the output byte moves with it one for one;
  * the same numbers through the NVFP4 loader (e4m3 scales 1.0, scale_2 =
    2^(s-127)) give the same planes;
  * byte 255 (NaN) makes the block invalid;
  * balancing: no effect on blocks without zeros; with zeros, the scale byte and
    the other codes are unchanged and the zeros' signs alternate; brute force
    with the option on, through both FP4 loaders;
  * the OpenMP build agrees bitwise.
"""
import random

import numpy as np
import pytest

import oracle
from oracle import tiny_exact
from bit_moe_expert_w2_gb300 import inputs

BAL = oracle.BALANCE_ZERO_SIGNS


def _nib(byts):
    return [(int(byts[i // 2]) >> (4 * (i % 2))) & 0xF for i in range(32)]


def _codes(code_bytes):
    return [(int(code_bytes[i // 4]) >> (2 * (i % 4))) & 3 for i in range(32)]


def _pack(nibs):
    b = np.zeros(16, np.uint8)
    for i, n in enumerate(nibs):
        b[i // 2] |= int(n) << (4 * (i % 2))
    return b


def _mx_block(nibs, s, options=0):
    c, u, st = oracle.requant_mxfp4(_pack(nibs).reshape(1, 1, 16), np.array([[[s]]], np.uint8), options=options)
    return _codes(c.reshape(-1)), int(u.reshape(-1)[0]), st


@pytest.mark.parametrize("s", [127, 118, 0, 1, 2, 253, 254])
def test_bruteforce_random_blocks_at_every_kind_of_scale(s):
    rnd = random.Random(100 + s)
    for _ in range(12):
        nibs = [rnd.randrange(16) for _ in range(32)]
        for bal in (0, BAL):
            codes, byte, st = _mx_block(nibs, s, bal)
            ref = tiny_exact.requant_block_mx(nibs, s, balance=bool(bal))
            assert st == 0 and (codes, byte) == (ref[0], ref[1]), (nibs, s, bal)


def test_bruteforce_few_distinct_values_and_zero_blocks():
    rnd = random.Random(7)
    cases = [[0] * 32, [8] * 32, [0, 8] * 16, [7] + [0] * 31, [1] + [0] * 31, [7] + [1] * 31, [6, 14] * 16]
    cases += [[rnd.choice([0, 8, 1, 9, 7, 15]) for _ in range(32)] for _ in range(10)]
    for nibs in cases:
        for s in (127, 1, 254):
            for bal in (0, BAL):
                codes, byte, st = _mx_block(nibs, s, bal)
                ref = tiny_exact.requant_block_mx(nibs, s, balance=bool(bal))
                assert st == 0 and (codes, byte) == (ref[0], ref[1]), (nibs, s, bal)


def test_codes_remap_shift_invariance():
    rng = np.random.default_rng(11)
    t = inputs.mxfp4_tensors(rng, 1, 64, 256)
    for d in (-40, -5, 3, 60):
        sc2 = (t.scales.astype(np.int32) + d).astype(np.uint8)
        c1, u1, st1 = oracle.requant_mxfp4(t.e2m1, t.scales)
        c2, u2, st2 = oracle.requant_mxfp4(t.e2m1, sc2)
        assert st1 == st2 == 0
        assert np.array_equal(c1, c2)
        assert np.array_equal(u2.astype(np.int32), u1.astype(np.int32) + d)


def test_same_numbers_through_the_nvfp4_loader():
    rng = np.random.default_rng(12)
    for s in (127, 100, 1, 200, 254):
        t = inputs.mxfp4_tensors(rng, 1, 8, 64)
        t.scales[:] = s
        e4m3_one = np.full((1, 8, 4), 0x38, np.uint8)   # 1.0
        s2 = np.array([np.ldexp(1.0, s - 127)], np.float32)
        for bal in (0, BAL):
            c1, u1, st1 = oracle.requant_mxfp4(t.e2m1, t.scales, options=bal)
            c2, u2, st2 = oracle.requant(t.e2m1, e4m3_one, s2, options=bal)
            assert st1 == st2 == 0 and np.array_equal(c1, c2) and np.array_equal(u1, u2), (s, bal)


def test_nan_scale_byte_is_invalid():
    codes, byte, st = _mx_block([3] * 32, 255)
    assert st == oracle.BAD_NVFP4 and byte == 0 and codes == [0] * 32
    assert tiny_exact.requant_block_mx([3] * 32, 255) is None


def test_balancing_changes_only_the_zeros_signs():
    rng = np.random.default_rng(13)
    t = inputs.plus_zero_nvfp4(rng, 2, 64, 256, zero_frac=0.3)
    c0, u0, st0 = oracle.requant(t.e2m1, t.e4m3, t.scale_2)
    c1, u1, st1 = oracle.requant(t.e2m1, t.e4m3, t.scale_2, options=BAL)
    assert st0 == st1 == 0 and np.array_equal(u0, u1)
    nib = np.stack([t.e2m1 & 0xF, t.e2m1 >> 4], axis=-1).reshape(2, 64, -1, 32)
    a = np.array([[_codes(b) for b in row.reshape(-1, 8)] for row in c0.reshape(-1, c0.shape[-1])]).reshape(nib.shape)
    b = np.array([[_codes(b) for b in row.reshape(-1, 8)] for row in c1.reshape(-1, c1.shape[-1])]).reshape(nib.shape)
    zero = (nib & 7) == 0
    assert zero.any() and (~zero).any()
    assert np.array_equal(a[~zero], b[~zero])
    assert ((a[zero] & 1) == 0).all() and ((b[zero] & 1) == 0).all()   # zeros sit at magnitude 1
    assert (a[zero] == 0).all()                                         # +0 -> +1 without the option
    rank = np.cumsum(zero, axis=-1) - 1                                 # j-th zero of its block
    assert np.array_equal(b[zero] >> 1, (rank[zero] & 1))


def test_balancing_bruteforce_nvfp4():
    rnd = random.Random(14)
    for _ in range(20):
        nibs = [rnd.choice([0, 0, 0, 8, 1, 2, 5, 7, 9, 15]) for _ in range(32)]
        pair = [rnd.choice([0x30, 0x38, 0x41, 0x00, 0xB8]) for _ in range(2)]
        s2 = float(np.float32(rnd.choice([2.0 ** -8, 0.75, 3e-3])))
        e2m1 = _pack(nibs).reshape(1, 1, 16)
        c, u, st = oracle.requant(e2m1, np.array(pair, np.uint8).reshape(1, 1, 2), np.array([s2], np.float32),
                                  options=BAL)
        ref = tiny_exact.requant_block(nibs, pair, s2, balance=True)
        assert st == 0 and (_codes(c.reshape(-1)), int(u.reshape(-1)[0])) == (ref[0], ref[1]), (nibs, pair, s2)


def test_parallel_build_agrees():
    rng = np.random.default_rng(15)
    t = inputs.mxfp4_tensors(rng, 3, 100, 512, plus_zero_frac=0.2)
    t.scales[1, 7, 3] = 255
    for bal in (0, BAL):
        a = oracle.requant_mxfp4(t.e2m1, t.scales, options=bal)
        b = oracle.requant_mxfp4(t.e2m1, t.scales, parallel=True, options=bal)
        assert all(np.array_equal(x, y) for x, y in zip(a[:2], b[:2])) and a[2] == b[2] == oracle.BAD_NVFP4
