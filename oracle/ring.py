"""Ring reduce-scatter / allreduce / allgather over k simulated ranks.

HOCCL (section 5, Limitations) leaves reduction collectives outside its
zero-SM scope and (section 6.1) falls back to NCCL for ReduceScatter, so the
pages fix neither the reduction order nor the rounding.  This oracle takes the
textbook ring reading:

* Block partition.  N elements per rank are split into k contiguous blocks;
  block r has B_r = floor(N/k) + [r < N mod k] elements and is owned by rank r.
* Ring.  ``order`` is a permutation of 0..k-1 (identity by default);
  succ(r) = order[(pos(r) + 1) mod k].  In ring reduce-scatter the partial sum
  of block r starts at succ(r), travels succ(r) -> succ^2(r) -> ... -> r, and
  every receiver adds its own input to the incoming partial.  So

      acc = x_{succ(r)}[blk r]
      acc = acc (+) x_{succ^j(r)}[blk r]   for j = 2 .. k     (succ^k(r) = r)
      y_r = narrow(acc)

* dtype rules.  float32: (+) is a binary32 add, round to nearest even, no
  flush-to-zero.  bfloat16: widen each operand exactly to binary32, add in
  binary32, round once to bf16 at the end ("fp32 accumulation").  int32: add
  modulo 2^32.
* ReduceScatter: rank r receives y_r.  AllReduce: every rank receives every
  y_r at block r's offset.  AllGather: rank r receives the concatenation of
  all ranks' sends (section 6.2, "AllGather").

bf16 arrays are uint16 bit patterns throughout.
"""
from __future__ import annotations

import numpy as np

from . import bf16 as _bf16

DTYPES = ("int32", "float32", "bfloat16")


def block_partition(n: int, k: int) -> tuple[list[int], list[int]]:
    """Sizes and offsets of the k owner blocks of an n-element rank buffer."""
    sizes = [n // k + (1 if r < n % k else 0) for r in range(k)]
    offs = [0] * k
    for r in range(1, k):
        offs[r] = offs[r - 1] + sizes[r - 1]
    return sizes, offs


def check_order(order, k: int) -> list[int]:
    if order is None:
        return list(range(k))
    order = [int(v) for v in order]
    if sorted(order) != list(range(k)):
        raise ValueError("ring order must be a permutation of 0..k-1")
    return order


def operand_sequence(r: int, order: list[int]) -> list[int]:
    """Ranks whose inputs block r folds, in ring order: succ(r), ..., succ^k(r)=r."""
    k = len(order)
    pos = order.index(r)
    return [order[(pos + j) % k] for j in range(1, k + 1)]


def _widen(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "float32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bfloat16":
        return _bf16.widen(x)
    if dtype == "int32":
        return np.asarray(x, dtype=np.int32).view(np.uint32)
    raise ValueError(dtype)


def _add(acc: np.ndarray, v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "int32":
        return (acc + v).astype(np.uint32)  # uint32 arithmetic wraps mod 2^32
    with np.errstate(invalid="ignore", over="ignore"):
        return np.add(acc, v, dtype=np.float32)


def _narrow(acc: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "float32":
        return acc.astype(np.float32)
    if dtype == "bfloat16":
        return _bf16.narrow(acc)
    return acc.astype(np.uint32).view(np.int32)


def fold(operands: list[np.ndarray], dtype: str) -> np.ndarray:
    """Left fold of equally long operand arrays in the given order, then narrow."""
    acc = _widen(operands[0], dtype).copy()
    for v in operands[1:]:
        acc = _add(acc, _widen(v, dtype), dtype)
    return _narrow(acc, dtype)


def reduce_block(xs: list[np.ndarray], r: int, lo: int, hi: int, dtype: str,
                 order: list[int]) -> np.ndarray:
    """y_r restricted to element range [lo, hi) of the rank buffers."""
    seq = operand_sequence(r, order)
    return fold([xs[j][lo:hi] for j in seq], dtype)


def allreduce(xs: list[np.ndarray], dtype: str, order=None) -> list[np.ndarray]:
    k = len(xs)
    order = check_order(order, k)
    n = len(xs[0])
    sizes, offs = block_partition(n, k)
    y = np.empty(n, dtype=np.asarray(xs[0]).dtype)
    for r in range(k):
        y[offs[r]:offs[r] + sizes[r]] = reduce_block(xs, r, offs[r], offs[r] + sizes[r], dtype, order)
    return [y.copy() for _ in range(k)]


def reduce_scatter(xs: list[np.ndarray], recvcount: int, dtype: str, order=None) -> list[np.ndarray]:
    """Each rank's input holds k * recvcount elements; rank r receives block r."""
    k = len(xs)
    order = check_order(order, k)
    for x in xs:
        if len(x) != k * recvcount:
            raise ValueError("reduce_scatter needs k * recvcount elements per rank")
    return [reduce_block(xs, r, r * recvcount, (r + 1) * recvcount, dtype, order) for r in range(k)]


def allgather(xs: list[np.ndarray]) -> list[np.ndarray]:
    y = np.concatenate([np.asarray(x) for x in xs])
    return [y.copy() for _ in range(len(xs))]


def sendrecv(x: np.ndarray) -> np.ndarray:
    """A point-to-point move delivers the sender's bytes unchanged."""
    return np.asarray(x).copy()


# The tolerance metric.  The workloads bound the result's error against a
# float64 naive sum (1e-6 for float32, 8e-3 for bfloat16); int32 results are
# compared bit for bit, so these functions take floating-point dtypes only.
def _check_float(dtype: str):
    if dtype not in TOL:
        raise ValueError(f"the tolerance metric is defined for {sorted(TOL)}, not {dtype}")


def naive_sum_f64(xs: list[np.ndarray], dtype: str) -> np.ndarray:
    """Elementwise float64 sum of all ranks (reference for the error bound)."""
    _check_float(dtype)
    acc = np.zeros(len(xs[0]), dtype=np.float64)
    for x in xs:
        acc += _widen(x, dtype).astype(np.float64)
    return acc


def abs_sum_f64(xs: list[np.ndarray], dtype: str) -> np.ndarray:
    _check_float(dtype)
    acc = np.zeros(len(xs[0]), dtype=np.float64)
    for x in xs:
        acc += np.abs(_widen(x, dtype).astype(np.float64))
    return acc


def normalized_error(y: np.ndarray, xs: list[np.ndarray], dtype: str) -> np.ndarray:
    """err_i = |y_i - s_i| / sum_r |x_{r,i}|; elements with a zero denominator
    must have y_i == 0 and then score 0 (else +inf)."""
    _check_float(dtype)
    s = naive_sum_f64(xs, dtype)
    d = abs_sum_f64(xs, dtype)
    yv = _widen(y, dtype).astype(np.float64)
    err = np.abs(yv - s)
    out = np.zeros_like(err)
    nz = d > 0
    out[nz] = err[nz] / d[nz]
    out[~nz] = np.where(yv[~nz] == 0, 0.0, np.inf)
    return out


# Tolerances of the path against the float64 naive sum (normalized error).
TOL = {"float32": 1e-6, "bfloat16": 8e-3}
