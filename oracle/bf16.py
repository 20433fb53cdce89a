"""bfloat16 <-> binary32 conversions written from the IEEE 754 definitions.

bfloat16 keeps the sign, the 8-bit exponent and the top 7 fraction bits of a
binary32 value.  Widening appends 16 zero fraction bits and is exact.
Narrowing rounds to the nearest representable bfloat16, ties to the neighbour
whose last fraction bit is 0 (round-to-nearest-even); NaN becomes a quiet NaN
with the sign kept.

Pinned in tests/test_oracle_bf16.py against PyTorch's CPU cast and against an
exact rational rounding (oracle.exact) on sampled bit patterns.
"""
from __future__ import annotations

import numpy as np


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> binary32 values, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def narrow(x: np.ndarray) -> np.ndarray:
    """binary32 values -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Let ``lo`` be the bf16 whose bits are the top 16 bits of x (x truncated
    toward zero) and ``hi`` the next bf16 away from zero (lo's pattern + 1).
    The low 16 bits ``rem`` of x measure the distance from lo in units of
    2^-16 of the gap lo->hi, so x is nearer lo when rem < 0x8000, nearer hi
    when rem > 0x8000, and halfway when rem == 0x8000, where the even pattern
    wins.  hi may be the infinity pattern 0x7F80 / 0xFF80: that is IEEE
    overflow (values at or past max + half an ulp round to infinity).
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lo = (u >> np.uint32(16)).astype(np.uint32)
    rem = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    lo_is_odd = (lo & np.uint32(1)) == 1
    take_hi = (rem > half) | ((rem == half) & lo_is_odd)
    out = np.where(take_hi, lo + np.uint32(1), lo)
    # NaN: exponent all ones and fraction non-zero -> quiet NaN, sign kept.
    is_nan = ((u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & ((u & np.uint32(0x007FFFFF)) != 0)
    sign = (u >> np.uint32(16)) & np.uint32(0x8000)
    out = np.where(is_nan, sign | np.uint32(0x7FC0), out)
    return out.astype(np.uint16)


def is_nan_bits(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
