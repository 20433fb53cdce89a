"""Helpers for the GPU parity tests: numpy <-> device tensors, guard bands."""
from __future__ import annotations

import numpy as np
import torch

NP = {"int32": np.int32, "float32": np.float32, "bfloat16": np.uint16, "uint8": np.uint8}
TORCH = {"int32": torch.int32, "float32": torch.float32, "bfloat16": torch.bfloat16, "uint8": torch.uint8}
ELEM = {"int32": 4, "float32": 4, "bfloat16": 2, "uint8": 1}
GUARD_BYTES = 4096
SENTINEL = 0xA5


def to_device(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bfloat16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach()
    if dtype == "bfloat16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bits(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype in (np.float32, np.int32):
        return a.view(np.uint32)
    return a


class Guarded:
    """A device buffer of `n` elements inside 4 KiB guard bands of 0xA5 bytes.

    ``offset_elems`` shifts the buffer inside the allocation to test
    misaligned pointers.  ``tensor`` is the usable view; ``check()`` asserts
    the guards are untouched.
    """

    def __init__(self, n: int, dtype: str, offset_elems: int = 0, fill: int = SENTINEL):
        b = ELEM[dtype]
        self.n, self.dtype = n, dtype
        self.lo = GUARD_BYTES + offset_elems * b
        self.raw = torch.full((self.lo + n * b + GUARD_BYTES,), fill, dtype=torch.uint8, device="cuda")
        self.raw[: self.lo].fill_(SENTINEL)
        self.raw[self.lo + n * b:].fill_(SENTINEL)
        self.tensor = self.raw[self.lo: self.lo + n * b].view(TORCH[dtype]) if n else self.raw[self.lo:self.lo].view(TORCH[dtype])

    def ptr(self) -> int:
        return self.raw.data_ptr() + self.lo

    def load(self, x: np.ndarray):
        self.tensor.copy_(to_device(x, self.dtype))

    def host(self) -> np.ndarray:
        return to_host(self.tensor, self.dtype)

    def check(self):
        lo = self.raw[: self.lo]
        hi = self.raw[self.lo + self.n * ELEM[self.dtype]:]
        assert bool((lo == SENTINEL).all()) and bool((hi == SENTINEL).all()), "guard band overwritten"


def assert_bits_equal(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    g, w = bits(got), bits(want)
    if dtype == "bfloat16":
        nan_w = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
        nan_g = ((g & 0x7F80) == 0x7F80) & ((g & 0x7F) != 0)
        assert np.array_equal(nan_w, nan_g), what
        g, w = g[~nan_w], w[~nan_w]
    if not np.array_equal(g, w):
        idx = np.nonzero(g != w)[0]
        raise AssertionError(f"{what}: {len(idx)} mismatches, first at {idx[:5]}: got {g[idx[:5]]} want {w[idx[:5]]}")
