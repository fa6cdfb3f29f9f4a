"""Independent binary32 arithmetic on rationals, used to pin the oracle.

Every operation is computed exactly with ``fractions.Fraction`` and then
rounded once to IEEE binary32 with round-to-nearest-even, including the
subnormal range, overflow to infinity and the IEEE sign-of-zero rules. It
does not use the host's float hardware for any rounding, so it checks the
oracle's compiled arithmetic (no contraction, a correctly rounded fmaf, no
flush-to-zero) from outside.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

_EMIN = -126          # smallest normal exponent
_P = 24               # significand bits
_MAX = (2 - Fraction(1, 1 << 23)) * (Fraction(2) ** 127)


def round_f32(q: Fraction, zero_sign: float = 1.0) -> float:
    """Round the rational ``q`` to binary32 (RNE); an exact zero gets ``zero_sign``."""
    if q == 0:
        return math.copysign(0.0, zero_sign)
    sign = -1.0 if q < 0 else 1.0
    a = -q if q < 0 else q
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, _EMIN)
    quantum = Fraction(2) ** (e - (_P - 1))
    scaled = a / quantum
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * quantum
    if r > _MAX:
        return sign * math.inf
    if r == 0:  # underflow to zero keeps the sign of the exact result
        return sign * 0.0
    return sign * float(r)


def _frac(x: float) -> Fraction:
    return Fraction(x)


def mul(a: float, b: float) -> float:
    if math.isnan(a) or math.isnan(b):
        return math.nan
    if math.isinf(a) or math.isinf(b):
        if a == 0 or b == 0:
            return math.nan
        return math.copysign(math.inf, math.copysign(1, a) * math.copysign(1, b))
    s = math.copysign(1, a) * math.copysign(1, b)
    return round_f32(_frac(a) * _frac(b), zero_sign=s)


def add(a: float, b: float) -> float:
    if math.isnan(a) or math.isnan(b):
        return math.nan
    if math.isinf(a) or math.isinf(b):
        if math.isinf(a) and math.isinf(b) and (a > 0) != (b > 0):
            return math.nan
        return a if math.isinf(a) else b
    both_neg_zero = (a == 0 and b == 0 and math.copysign(1, a) < 0 and math.copysign(1, b) < 0)
    return round_f32(_frac(a) + _frac(b), zero_sign=-1.0 if both_neg_zero else 1.0)


def fma(a: float, b: float, c: float) -> float:
    if math.isnan(a) or math.isnan(b) or math.isnan(c):
        return math.nan
    if math.isinf(a) or math.isinf(b):
        if a == 0 or b == 0:
            return math.nan
        p = math.copysign(math.inf, math.copysign(1, a) * math.copysign(1, b))
        if math.isinf(c) and (c > 0) != (p > 0):
            return math.nan
        return p
    if math.isinf(c):
        return c
    exact = _frac(a) * _frac(b) + _frac(c)
    if exact == 0:
        # Zero product plus zero addend keeps a shared sign; an exact
        # cancellation of non-zero terms is +0 under round-to-nearest.
        if (a == 0 or b == 0) and c == 0:
            ps = math.copysign(1, a) * math.copysign(1, b)
            return -0.0 if (ps < 0 and math.copysign(1, c) < 0) else 0.0
        return 0.0
    return round_f32(exact)


def canonical_bits(v: float) -> int:
    if math.isnan(v):
        return 0x7FC00000
    return int(np.float32(v).view(np.uint32))


def gemm_bits(A: np.ndarray, B: np.ndarray, mode: int) -> np.ndarray:
    """Output bits of the pages' per-output loop, on this module's arithmetic."""
    m, k = A.shape
    n = B.shape[1]
    out = np.zeros((m, n), dtype=np.uint32)
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for p in range(k):
                a, b = float(A[i, p]), float(B[p, j])
                acc = fma(a, b, acc) if mode == 1 else add(acc, mul(a, b))
            out[i, j] = canonical_bits(acc)
    return out
