"""Exact rational arithmetic for pinning the oracle's floating point.

Independent of the oracle's C code: values are Python Fractions and rounding
to a binary format is done from its definition (nearest representable value,
ties to the even significand) with Python integers.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

INF = float("inf")


def f32_bits_to_fraction(bits: int) -> Fraction:
    v = struct.unpack("<f", struct.pack("<I", bits & 0xFFFFFFFF))[0]
    assert math.isfinite(v)
    return Fraction(v)


def round_binary(q: Fraction, mant_bits: int, emin: int, emax: int):
    """Round q to the binary format with `mant_bits` significand bits
    (including the implicit one), normal exponents [emin, emax], gradual
    underflow. Returns a Fraction, or +-inf on overflow."""
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (mant_bits - 1))
    n = a / quantum
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    r = lo * quantum
    if r >= Fraction(2) ** (emax + 1):
        return sign * INF
    return sign * r


def round_f32(q: Fraction):
    return round_binary(q, 24, -126, 127)


def round_bf16(q: Fraction):
    return round_binary(q, 8, -126, 127)


def bf16_bits(v) -> int:
    """BF16 bit pattern of an exactly representable value (Fraction or inf)."""
    if v == INF:
        return 0x7F80
    if v == -INF:
        return 0xFF80
    f = float(v)
    bits = struct.unpack("<I", struct.pack("<f", f))[0]
    assert bits & 0xFFFF == 0, "value is not a BF16 number"
    return bits >> 16
