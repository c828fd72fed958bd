"""Exact-rational helpers for pinning the oracle (no numpy/C float arithmetic).

Values are Python Fractions; rounding to a binary format is done with integer
arithmetic, round-to-nearest, ties-to-even, for a format with ``p`` significand
bits (24 for binary32, 8 for bf16) and minimum normal exponent -126 (both).
"""
from fractions import Fraction
import struct

import numpy as np


def f32_exact(v) -> Fraction:
    return Fraction(float(np.float32(v)))


def bf16_bits_exact(b: int) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<I", (int(b) & 0xFFFF) << 16))[0])


def round_rne(q: Fraction, p: int, emin: int = -126) -> Fraction:
    """Round q to the nearest value with p significand bits (ties to even),
    exponent >= emin for normals, gradual underflow below.  No overflow."""
    if q == 0:
        return Fraction(0)
    s = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (p - 1))
    m = a / ulp
    n = m.numerator // m.denominator
    r = m - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * n * ulp


def to_f32(q: Fraction) -> np.float32:
    r = round_rne(q, 24)
    return np.float32(float(r))  # exact: r is representable in binary32


def to_bf16_bits(q: Fraction) -> int:
    r = round_rne(q, 8)
    f = np.float32(float(r))
    return int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)
