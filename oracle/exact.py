"""Exact rational arithmetic helpers for the oracle (test infrastructure only).

Everything here works on Python integers, so results are exact and do not
depend on summation order.  They serve two readings of the pages' silent
points:

* the double-quantisation mean ``mu`` of the block absmax constants is the
  exact arithmetic mean, rounded once to the nearest fp32 (ties to even);
* conversion of an fp32 value to bf16 rounds to nearest, ties to even.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

F32_MIN_EXP = -126  # exponent of the smallest normal fp32
F32_MANT = 23       # explicit mantissa bits of fp32


def f32_to_fraction(x: np.float32) -> Fraction:
    """Exact rational value of a finite fp32."""
    return Fraction(float(np.float32(x)))


def exact_sum_f32(values: np.ndarray) -> Fraction:
    """Exact sum of finite, non-negative fp32 values, as a Fraction.

    Each value is split into its integer significand ``M`` and its exponent
    field ``e``: value = M * 2**(max(e,1) - 150).  Significands are summed
    exactly per exponent (int64 cannot overflow: M < 2**24 and at most 2**39
    terms share an exponent), and the per-exponent sums are combined with
    Python's unbounded integers.
    """
    v = np.ascontiguousarray(values, dtype=np.float32)
    if v.size == 0:
        return Fraction(0)
    if np.any(v < 0) or not np.all(np.isfinite(v)):
        raise ValueError("exact_sum_f32 expects finite non-negative values")
    bits = v.view(np.uint32).astype(np.int64)
    e = (bits >> 23) & 0xFF
    mant = bits & 0x7FFFFF
    sig = mant + np.where(e > 0, 1 << 23, 0)
    ep = np.maximum(e, 1)
    total = 0
    for ex in np.unique(ep):
        s = int(sig[ep == ex].sum(dtype=np.int64))
        total += s << int(ex - 1)  # value * 2**149 = M * 2**(e'-1)
    return Fraction(total, 1 << 149)


def round_fraction_to_f32(x: Fraction) -> np.float32:
    """Nearest fp32 to the exact rational ``x`` (ties to even, subnormals kept).

    Finds the binade of |x|, takes the unit in the last place of that binade
    (2**-149 below the normal range), divides, and rounds the integer
    quotient half-to-even.  Overflow beyond the largest finite fp32 raises.
    """
    if x == 0:
        return np.float32(0.0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    num, den = a.numerator, a.denominator
    # E = floor(log2(a))
    E = num.bit_length() - den.bit_length()
    if Fraction(2) ** E > a:
        E -= 1
    elif Fraction(2) ** (E + 1) <= a:
        E += 1
    q_exp = max(E, F32_MIN_EXP) - F32_MANT  # exponent of one ulp
    scaled = a / (Fraction(2) ** q_exp)
    f = scaled.numerator // scaled.denominator
    rem = scaled - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    value = f * (2.0 ** q_exp)  # exact in float64: f <= 2**24
    if value > float(np.finfo(np.float32).max):
        raise OverflowError("value exceeds the fp32 range")
    return np.float32(sign * value)


def exact_mean_f32(values: np.ndarray) -> np.float32:
    """Exact arithmetic mean of non-negative fp32 values, rounded once to fp32."""
    v = np.asarray(values, dtype=np.float32)
    if v.size == 0:
        return np.float32(0.0)
    return round_fraction_to_f32(exact_sum_f32(v) / v.size)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    A bf16 keeps the upper 16 bits of an fp32.  The discarded lower half is
    compared with one half-ulp (0x8000): above it rounds up, below it rounds
    down, and exactly at it the result is the neighbour whose last kept bit
    is 0.  Finite inputs only.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi = b >> 16
    lo = b & 0xFFFF
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    return (hi + up.astype(np.uint64)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)
