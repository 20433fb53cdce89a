"""Seeded synthetic inputs for the five collective workloads.

This module only draws random numbers and lays them out; it holds none of the
collective arithmetic (no reduction, no copy schedule, no rounding rule of the
method).  Both the CPU oracle tests and the GPU path take their inputs from
here, so the two sides see identical bytes.

Conventions
-----------
* Every generator is ``numpy.random.default_rng(seed)`` (PCG64).
* The workload on 4 ranks of 1,048,576 fp32 values uses seed ``r`` for rank
  ``r``.  Every other workload uses ``1000 * workload + 100 * slot + r``.
* bf16 tensors are returned as ``uint16`` bit patterns.  They are drawn in
  float32 and converted to bfloat16 by PyTorch's CPU cast (round to nearest,
  ties to even), a library routine used here only to produce input bytes.
"""
from __future__ import annotations

import numpy as np

# Workload sizes (the five workloads of the DP / PP / EP evaluation mix).
AR_SMALL = dict(k=4, n=1_048_576, dtype="float32", chunks=4)
AR_LARGE = dict(k=8, n=134_217_728, dtype="bfloat16", sigma=1e-3)
RS_BUCKETS = dict(k=8, buckets=268, bucket_elems=13_107_200, dtype="bfloat16",
                  sigma=1e-3, pool=16)
PP_STAGES = dict(p=8, microbatches=16, seq=4096, hidden=4096, dtype="bfloat16")
EP_DISPATCH = dict(k=8, tokens=4096, hidden=2048, experts=64, topk=6, zipf=1.1)


def seed_for(workload: int, slot: int, rank: int) -> int:
    return 1000 * workload + 100 * slot + rank


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Library cast float32 -> bfloat16 bits (input preparation only)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def uniform_f32(n: int, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.uniform(lo, hi, size=n).astype(np.float32)


def normal_f32(n: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=n, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    return x


def normal_bf16(n: int, seed: int, sigma: float = 1.0) -> np.ndarray:
    return f32_to_bf16_bits(normal_f32(n, seed, sigma))


def uniform_i32(n: int, seed: int, lo: int = -(2 ** 30), hi: int = 2 ** 30) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, size=n, dtype=np.int64, endpoint=True).astype(np.int32)


def rank_inputs(dtype: str, k: int, n: int, workload: int = 0, slot: int = 0,
                sigma: float = 1.0) -> list[np.ndarray]:
    """One input vector per simulated rank.

    ``float32``: uniform[-1, 1]; ``bfloat16``: N(0, sigma) as bf16 bits;
    ``int32``: uniform integers in [-2^30, 2^30] (sums of 8 wrap around).
    """
    out = []
    for r in range(k):
        s = r if workload == 1 else seed_for(workload, slot, r)
        if dtype == "float32":
            out.append(uniform_f32(n, s))
        elif dtype == "bfloat16":
            out.append(normal_bf16(n, s, sigma))
        elif dtype == "int32":
            out.append(uniform_i32(n, s))
        else:
            raise ValueError(dtype)
    return out


def small_int_inputs(dtype: str, k: int, n: int, seed: int, bound: int) -> list[np.ndarray]:
    """Integer-valued inputs whose sums are exact in every order (|x| <= bound)."""
    rng = np.random.default_rng(seed)
    vals = [rng.integers(-bound, bound, size=n, endpoint=True) for _ in range(k)]
    if dtype == "float32":
        return [v.astype(np.float32) for v in vals]
    if dtype == "bfloat16":
        return [f32_to_bf16_bits(v.astype(np.float32)) for v in vals]
    if dtype == "int32":
        return [v.astype(np.int32) for v in vals]
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# Pipeline-parallel workload: per-(stage, micro-batch, direction) XOR keys.
# ---------------------------------------------------------------------------
def pp_keys(p: int, m: int, seed: int = 4000) -> np.ndarray:
    """Non-zero 16-bit keys, shape [p, m, 2] (direction 0 = forward, 1 = backward)."""
    rng = np.random.default_rng(seed)
    return rng.integers(1, 1 << 16, size=(p, m, 2), dtype=np.int64).astype(np.uint16)


def pp_activations(m: int, elems: int, seed_base: int = 4100) -> list[np.ndarray]:
    """Micro-batch activations, N(0, 1) as bf16 bits, one array per micro-batch."""
    return [normal_bf16(elems, seed_base + i) for i in range(m)]


# ---------------------------------------------------------------------------
# Expert-parallel workload: Zipf(1.1) routing over 64 experts, top-6.
# ---------------------------------------------------------------------------
def zipf_probs(experts: int, s: float) -> np.ndarray:
    w = (np.arange(experts, dtype=np.float64) + 1.0) ** (-s)
    return w / w.sum()


def ep_routing(k: int, tokens: int, experts: int, topk: int, s: float,
               seed_base: int = 5000) -> list[np.ndarray]:
    """Per source rank, an int array [tokens, topk] of distinct expert ids.

    Expert ids are drawn without replacement from the bounded Zipf law
    p(e) ~ (e+1)^-s; experts 8r..8r+7 live on rank r (experts // (experts/k)).
    """
    p = zipf_probs(experts, s)
    out = []
    for r in range(k):
        rng = np.random.default_rng(seed_base + r)
        rows = np.empty((tokens, topk), dtype=np.int64)
        for t in range(tokens):
            rows[t] = rng.choice(experts, size=topk, replace=False, p=p)
        out.append(rows)
    return out


def ep_token_rows(k: int, tokens: int, hidden: int, seed_base: int = 5000) -> list[np.ndarray]:
    """Per source rank, the token rows [tokens, hidden] as bf16 bits, N(0, 1)."""
    return [normal_bf16(tokens * hidden, seed_base + 500 + r).reshape(tokens, hidden) for r in range(k)]
