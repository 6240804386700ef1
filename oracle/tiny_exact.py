"""Exact rational brute force for small requant cases (Python Fractions).

TEST INFRASTRUCTURE ONLY.  Independent of ``oracle.c``: it follows the plain
definition with no candidate window and no integer tricks.

Definition followed (page "The v0.24.0 port", section "Our hooks", modelopt.py,
fp8.py and mxfp4.py bullets; page "vLLM-Moet wiki", section "2-bit expert
planes"): each NVFP4 element is e2m1 x e4m3 x scale_2, each FP8 element e4m3 x
its f32 128 x 128 block scale and each MXFP4 element e2m1 x 2^(s-127), an
exact rational number; a block of 32 is
re-quantized to codes from {-4,-1,1,4} times one UE8M0 scale 2^u, u in
[-126,125], minimising the squared error.  With the scale fixed the error
separates per element, so for every u each element takes its nearest code;
exact ties between codes go to magnitude 1, exact ties between scales to the
smaller u, and the code's sign is the element's sign bit.  With zero-sign
balancing (page "vLLM-Moet wiki", the Kimi-K2.7 paragraph) the exact zeros of
the block take the signs +,-,+,- ... in element order instead.
"""
from __future__ import annotations

from fractions import Fraction

E2M1_MAGNITUDES = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
                   Fraction(2), Fraction(3), Fraction(4), Fraction(6)]


def e2m1(nib: int):
    """(negative?, |value|) of an e2m1 nibble: 1 sign, 2 exponent, 1 mantissa bit."""
    nib = int(nib)
    sign = (nib >> 3) & 1
    e, m = (nib >> 1) & 3, nib & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return bool(sign), mag


def e4m3(b: int):
    """(negative?, |value|) of an e4m3fn byte, or None for NaN."""
    b = int(b)
    sign = (b >> 7) & 1
    e, m = (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return None
    mag = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return bool(sign), mag


def f32(v: float) -> Fraction:
    return Fraction(v)


def requant_block(nibbles, e4m3_pair, scale_2: float, balance: bool = False):
    """nibbles: 32 ints; e4m3_pair: 2 bytes; -> (codes[32], scale byte) or None when invalid."""
    sc = [e4m3(b) for b in e4m3_pair]
    if any(s is None for s in sc) or not (scale_2 > 0) or scale_2 == float("inf"):
        return None
    s2 = f32(scale_2)
    neg, mag = [], []
    for i, nib in enumerate(nibbles):
        n_neg, n_mag = e2m1(nib)
        s_neg, s_mag = sc[i // 16]
        neg.append(n_neg != s_neg)
        mag.append(n_mag * s_mag * s2)
    return _search(neg, mag, balance)


def requant_block_mx(nibbles, scale_byte: int, balance: bool = False):
    """MXFP4: 32 e2m1 nibbles under one UE8M0 byte -> (codes[32], scale byte), or None for byte 255."""
    if int(scale_byte) == 255:
        return None
    step = Fraction(2) ** (int(scale_byte) - 127)
    vals = [e2m1(n) for n in nibbles]
    return _search([n for n, _ in vals], [m * step for _, m in vals], balance)


def _search(neg, mag, balance: bool = False):
    """(codes[32], scale byte) minimising the exact squared error over all u."""
    if balance:
        neg, z = list(neg), 0
        for i, a in enumerate(mag):
            if a == 0:
                neg[i] = bool(z & 1)
                z += 1
    best = None
    for u in range(-126, 126):
        step = Fraction(2) ** u
        sse = Fraction(0)
        for a in mag:
            v = 4 * step if a > Fraction(5, 2) * step else step
            sse += (a - v) ** 2
        if best is None or sse < best[0]:
            best = (sse, u)
    u = best[1]
    step = Fraction(2) ** u
    codes = [(int(n) << 1) | (1 if a > Fraction(5, 2) * step else 0) for n, a in zip(neg, mag)]
    return codes, u + 127


def requant_block_fp8(e4m3_bytes, scale: float):
    """32 e4m3fn bytes under one f32 block scale -> (codes[32], scale byte), or None when invalid."""
    if not (scale > 0) or scale == float("inf"):
        return None
    vals = [e4m3(b) for b in e4m3_bytes]
    if any(v is None for v in vals):
        return None
    s = f32(scale)
    return _search([n for n, _ in vals], [m * s for _, m in vals])


def nearest_codes_by_enumeration(values, u: int):
    """Exhaustive argmin over all 4^n code vectors at a fixed scale (ties: first
    vector in the order that prefers magnitude 1, then the element's own sign)."""
    import itertools
    step = Fraction(2) ** u
    levels = {0: step, 1: 4 * step, 2: -step, 3: -4 * step}
    best = None
    for combo in itertools.product(range(4), repeat=len(values)):
        sse = sum((v - levels[c]) ** 2 for v, c in zip(values, combo))
        key = (sse, tuple((c & 1) for c in combo))
        if best is None or key < best[0]:
            best = (key, combo)
    return list(best[1]), best[0][0]
