"""Pins of the bf16 conversions (CPU only)."""
import numpy as np

from oracle import bf16
from tests import pins


def test_narrow_matches_library_cast():
    pins.check_bf16_narrow_vs_torch(bf16.narrow, np.random.default_rng(0))


def test_narrow_matches_exact_rounding():
    pins.check_bf16_narrow_exact(bf16.narrow, np.random.default_rng(1))


def test_widen_is_exact_and_roundtrips():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    w = bf16.widen(b)
    assert np.array_equal(w.view(np.uint32) >> 16, b.astype(np.uint32))
    assert np.array_equal(w.view(np.uint32) & 0xFFFF, np.zeros(1 << 16, np.uint32))
    back = bf16.narrow(w)
    nan = bf16.is_nan_bits(b)
    assert np.array_equal(back[~nan], b[~nan])
    assert bf16.is_nan_bits(back[nan]).all()
