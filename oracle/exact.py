"""Exact rational arithmetic and correctly rounded binary32 / bfloat16.

Used only by the pins in tests/: it rounds exact rationals to the nearest
binary32 (or bfloat16) by the definition -- scale into the target's
significand range, round the scaled rational to an integer with ties to even,
handle the subnormal range and overflow -- without touching any floating-point
hardware path.
"""
from __future__ import annotations

import struct
from fractions import Fraction


def f32_bits_to_fraction(bits: int) -> Fraction | None:
    """Exact value of a binary32 bit pattern; None for Inf/NaN."""
    sign = -1 if bits >> 31 else 1
    e = (bits >> 23) & 0xFF
    f = bits & 0x7FFFFF
    if e == 0xFF:
        return None
    if e == 0:
        return sign * Fraction(f, 1 << 149)
    return sign * Fraction((1 << 23) | f) * Fraction(2) ** (e - 150)


def float32_to_fraction(x) -> Fraction:
    bits = struct.unpack("<I", struct.pack("<f", float(x)))[0]
    v = f32_bits_to_fraction(bits)
    if v is None:
        raise ValueError("not finite")
    return v


def _round_half_even(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2):
        return fl + 1
    if rem < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def round_to_format(v: Fraction, mant_bits: int, emin: int, emax: int) -> tuple[int, int, int] | str:
    """Nearest value of a binary format with ``mant_bits`` stored fraction bits.

    Returns (sign, biased_exponent, fraction) or the string 'inf' / '-inf'.
    emin / emax are the unbiased exponents of the normal range.
    """
    sign = 1 if v < 0 else 0
    a = -v if v < 0 else v
    if a == 0:
        return (sign, 0, 0)
    p = mant_bits + 1
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)                      # subnormals share the emin scale
    m = _round_half_even(a / Fraction(2) ** (e - p + 1))
    if m == 1 << p:                       # rounding carried into the next binade
        m >>= 1
        e += 1
    if e > emax:
        return "-inf" if sign else "inf"
    if m < (1 << (p - 1)):                # subnormal (or zero)
        return (sign, 0, m)
    bias = emax                           # IEEE bias equals emax
    return (sign, e + bias, m - (1 << (p - 1)))


def round_to_f32_bits(v: Fraction) -> int:
    r = round_to_format(v, 23, -126, 127)
    if r == "inf":
        return 0x7F800000
    if r == "-inf":
        return 0xFF800000
    s, e, f = r
    return (s << 31) | (e << 23) | f


def round_to_bf16_bits(v: Fraction) -> int:
    r = round_to_format(v, 7, -126, 127)
    if r == "inf":
        return 0x7F80
    if r == "-inf":
        return 0xFF80
    s, e, f = r
    return (s << 15) | (e << 7) | f


def exact_ring_fold_f32(operands: list[int]) -> int:
    """Fold binary32 bit patterns left to right, each add rounded exactly once.

    The sign of an exact zero is not tracked (an exact zero sum is +0, the
    IEEE round-to-nearest result for x + (-x)); callers avoid -0 + -0.
    """
    acc = f32_bits_to_fraction(operands[0])
    bits = operands[0]
    for b in operands[1:]:
        v = f32_bits_to_fraction(b)
        bits = round_to_f32_bits(acc + v)
        acc = f32_bits_to_fraction(bits)
    return bits
