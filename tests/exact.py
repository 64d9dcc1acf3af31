"""Exact rational arithmetic used to pin the oracle's floating point.

Independent of the oracle: values are decoded from their IEEE bit patterns
into ``fractions.Fraction`` and rounded back with round-to-nearest, ties to
even, by comparing against the two neighbouring representable values.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def f32_from_bits(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def frac_of_f32(x: float) -> Fraction:
    """Exact value of a finite float32 (Python float holds it exactly)."""
    assert math.isfinite(x)
    return Fraction(x)


def frac_of_bf16(b: int) -> Fraction:
    return Fraction(f32_from_bits((b & 0xFFFF) << 16))


def round_binary(v: Fraction, p: int, emin: int, emax: int):
    """Round an exact value to a binary format with p significand bits,
    minimum normal exponent emin and maximum exponent emax, to nearest with
    ties to even.  Returns (sign, Fraction magnitude) or (sign, inf)."""
    sign = -1 if v < 0 else 1
    a = -v if v < 0 else v
    if a == 0:
        return sign, Fraction(0)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)                      # subnormal range shares emin's spacing
    ulp = Fraction(2) ** (e - (p - 1))
    q, r = divmod(a, ulp)
    q = int(q)
    half = ulp / 2
    rem = a - q * ulp
    if rem > half or (rem == half and q % 2 == 1):
        q += 1
    mag = q * ulp
    max_finite = (2 - Fraction(2) ** (1 - p)) * Fraction(2) ** emax
    if mag > max_finite:
        return sign, math.inf
    return sign, mag


def round_f32(v: Fraction) -> float:
    s, m = round_binary(v, 24, -126, 127)
    if m == math.inf:
        return s * math.inf
    out = float(m)                        # exact: m is a float32 value
    return -out if s < 0 else (out if m != 0 else (0.0 if s > 0 else -0.0))


def round_bf16_bits(v: Fraction, neg_zero: bool = False) -> int:
    """bf16 bit pattern of the correctly rounded value of v."""
    s, m = round_binary(v, 8, -126, 127)
    if m == math.inf:
        u = 0x7F800000
    else:
        u = f32_bits(float(m))
        assert u & 0xFFFF == 0
    if s < 0 or (m == 0 and neg_zero):
        u |= 0x80000000
    return u >> 16


def fma_f32(a: float, b: float, c: float) -> float:
    """IEEE fused multiply-add of float32 values, exactly rounded once.
    Zero results take the sign the IEEE rules give in round-to-nearest."""
    v = frac_of_f32(a) * frac_of_f32(b) + frac_of_f32(c)
    if v == 0:
        prod_neg = (math.copysign(1, a) * math.copysign(1, b)) < 0
        prod_zero = (a == 0 or b == 0)
        if prod_zero and c == 0:
            # exact zero sum of two zeros: negative only if both are negative
            return -0.0 if (prod_neg and math.copysign(1, c) < 0) else 0.0
        return 0.0
    return round_f32(v)


def bf16_of_f32(x: float) -> int:
    """RNE float32 -> bf16 bits (finite inputs and +-inf)."""
    if math.isinf(x):
        return 0xFF80 if x < 0 else 0x7F80
    if x == 0:
        return 0x8000 if math.copysign(1, x) < 0 else 0
    return round_bf16_bits(frac_of_f32(x))
