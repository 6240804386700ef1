"""Pins for the oracle's value tables (CPU only).

e2m1 and e4m3fn are checked exhaustively against their bit-field definitions in
exact rationals; the codebook against the set the pages print ({-4,-1,1,4},
page "vLLM-Moet wiki", section "2-bit expert planes"), including the pages'
claim that it is exact in e2m1 and bf16; the bf16 rounding against an exact
nearest-even rounding done with Fractions.
"""
import math
import random
from fractions import Fraction

import numpy as np

import oracle


def test_e2m1_all_nibbles():
    # 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal.
    expected_mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    for nib in range(16):
        v = oracle.e2m1_value(nib)
        assert abs(v) == expected_mags[nib & 7]
        assert math.copysign(1.0, v) == (-1.0 if nib & 8 else 1.0)


def _e4m3_fraction(b):
    s, e, m = b >> 7, (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return None
    mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def test_e4m3_all_bytes():
    for b in range(256):
        ref = _e4m3_fraction(b)
        v = oracle.e4m3_value(b)
        if ref is None:
            assert math.isnan(v)
        else:
            assert Fraction(v) == ref
    assert oracle.e4m3_value(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_codebook_is_sign_symmetric_and_exact_in_e2m1_and_bf16():
    vals = sorted(oracle.code_value(c) for c in range(4))
    assert vals == [-4.0, -1.0, 1.0, 4.0]
    e2m1_vals = {oracle.e2m1_value(n) for n in range(16)}
    for v in vals:
        assert v in e2m1_vals
        assert oracle.bf16_to_double(oracle.bf16_from_double(v)) == v
    # negation is the sign bit of the code (reading R1)
    for c in range(4):
        assert oracle.code_value(c ^ 2) == -oracle.code_value(c)


def _bf16_round_exact(v: float) -> float:
    """Nearest bf16 (8 significant bits, subnormal quantum 2^-133), ties to even."""
    if v == 0:
        return v
    a = Fraction(abs(v))
    e = math.frexp(abs(v))[1] - 1
    q = e - 7 if e >= -126 else -133
    step = Fraction(2) ** q
    lo = (a // step) * step
    hi = lo + step
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if ((lo / step) % 2 == 0) else hi
    if r > Fraction(2) ** 127 * (2 - Fraction(1, 128)):
        return math.copysign(math.inf, v)
    return math.copysign(float(r), v)


def test_bf16_rounding_random_and_ties():
    rnd = random.Random(7)
    cases = [1.0, -1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -40, 3.0e38, 3.4e38,
             2.0 ** -130, 2.0 ** -133 * 1.5, 2.0 ** -133 * 2.5, 1e-45, 0.1, -0.7310585786300049]
    cases += [rnd.uniform(-10, 10) * 2.0 ** rnd.randint(-140, 120) for _ in range(3000)]
    for v in cases:
        got = oracle.bf16_to_double(oracle.bf16_from_double(v))
        assert got == _bf16_round_exact(v) or (math.isinf(got) and math.isinf(_bf16_round_exact(v))), v


def test_bf16_bits_roundtrip_matches_numpy():
    bits = np.arange(0, 65536, 37, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    for b, v in zip(bits[:500], f[:500]):
        if np.isnan(v):
            continue
        assert oracle.bf16_to_double(int(b)) == float(v)
