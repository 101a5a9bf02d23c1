"""Exact rational bf16 arithmetic for pinning the oracle.

Written from the IEEE-754 field definitions (1 sign bit, 8 exponent bits with
bias 127, 7 fraction bits; exponent field 0 = subnormal/zero, 255 = inf/NaN)
with Python Fractions, so it shares neither code nor method with the oracle's
C (which widens by bit shift and rounds with rint on a scaled double).
"""
from __future__ import annotations

from fractions import Fraction

BIAS = 127
FRAC_BITS = 7
MIN_NORMAL_EXP = 1 - BIAS          # 2^-126
SUBNORMAL_QUANTUM = Fraction(1, 2 ** (BIAS - 1 + FRAC_BITS))  # 2^-133
OVERFLOW = Fraction(2) ** 128


def value(bits: int):
    """Exact value of a bf16 bit pattern: Fraction, or float inf/nan."""
    bits &= 0xFFFF
    sign = -1 if bits >> 15 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        return float("nan") if f else sign * float("inf")
    if e == 0:
        return sign * f * SUBNORMAL_QUANTUM
    return sign * (1 + Fraction(f, 2 ** FRAC_BITS)) * Fraction(2) ** (e - BIAS)


def _binade(a: Fraction) -> int:
    """The e with 2^e <= a < 2^(e+1), for a > 0, by exact comparisons."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def encode(v: Fraction, negative: bool) -> int:
    """Bits of an exactly representable bf16 magnitude v >= 0."""
    sign = 0x8000 if negative else 0
    if v == 0:
        return sign
    e = _binade(v)
    if e >= MIN_NORMAL_EXP:
        frac = (v / Fraction(2) ** e - 1) * 2 ** FRAC_BITS
        assert frac.denominator == 1 and 0 <= frac < 128, v
        return sign | ((e + BIAS) << 7) | int(frac)
    frac = v / SUBNORMAL_QUANTUM
    assert frac.denominator == 1 and 0 < frac < 128, v
    return sign | int(frac)


def round_bf16(x) -> int:
    """Round an exact rational (or int) to bf16 bits, nearest, ties to even."""
    x = Fraction(x)
    neg = x < 0
    a = -x if neg else x
    if a == 0:
        return 0x8000 if neg else 0
    e = _binade(a)
    quantum = max(Fraction(2) ** (e - FRAC_BITS), SUBNORMAL_QUANTUM)
    scaled = a / quantum
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * quantum
    if r >= OVERFLOW:
        return (0x8000 if neg else 0) | 0x7F80
    return encode(r, neg)
