"""Expert-parallel pack (dispatch side) and combine (unpack) around the all-to-all.

HOCCL names EP token dispatch / combine as all-to-all traffic (section 2.1,
Table 1); the exchange itself is oracle.alltoall.  What surrounds it:

pack: the rows of source rank s are its (token, slot) pairs, one per chosen
  expert, ordered by (destination rank, expert, token, slot); experts
  e = 0..E-1 live on rank e // (E / k), so the order is by expert, then token,
  then slot.  Row i of the send buffer is the token row x[token_i]; perm[i] is
  token_i * topk + slot_i and pos_of is its inverse; dst_counts[d] = the number
  of rows for rank d times `hidden` (elements).

combine: after the inverse exchange every source rank holds its rows back in
  packed order; token t's output is the gate-weighted sum of its topk rows,
      prod_j = fp32(w[t, j] * row[pos_of[t*topk + j]])    (binary32 product, RNE)
      y[t]   = bf16( ((prod_0 + prod_1) + prod_2) + ... ) (binary32 adds, one final rounding)
  folded in slot order, no fused multiply-add.

Pairs whose expert id lies outside [0, E) are dropped: they get no row, their
pos_of is -1 and the combine skips them (a token with no valid slot gets +0).

bf16 arrays are uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np

from . import bf16 as _bf16


def pack_order(expert_ids: np.ndarray, experts: int) -> np.ndarray:
    """perm: flattened (token, slot) indices of the valid pairs in (expert, token, slot) order."""
    flat = np.asarray(expert_ids).reshape(-1)
    valid = np.nonzero((flat >= 0) & (flat < experts))[0]
    return valid[np.argsort(flat[valid], kind="stable")].astype(np.int64)


def pack(x_bits: np.ndarray, expert_ids: np.ndarray, experts: int, k: int):
    """Returns (send rows [valid pairs, H], perm, pos_of, dst_counts in elements)."""
    tokens, topk = expert_ids.shape
    hidden = x_bits.shape[1]
    perm = pack_order(expert_ids, experts)
    pos_of = np.full(tokens * topk, -1, dtype=np.int64)
    pos_of[perm] = np.arange(len(perm))
    send = x_bits[perm // topk]
    per_rank = experts // k
    flat = expert_ids.reshape(-1)
    dst = flat[perm] // per_rank
    counts = np.bincount(dst, minlength=k).astype(np.int64) * hidden
    return np.ascontiguousarray(send), perm, pos_of, counts


def combine(rows_bits: np.ndarray, pos_of: np.ndarray, weights: np.ndarray, topk: int) -> np.ndarray:
    tokens = len(pos_of) // topk
    hidden = rows_bits.shape[1]
    w = np.asarray(weights, dtype=np.float32).reshape(tokens, topk)
    pos = np.asarray(pos_of).reshape(tokens, topk)
    acc = np.zeros((tokens, hidden), dtype=np.float32)
    seen = np.zeros(tokens, dtype=bool)
    for j in range(topk):
        ok = pos[:, j] >= 0
        r = _bf16.widen(rows_bits[np.where(ok, pos[:, j], 0)])
        with np.errstate(invalid="ignore", over="ignore"):
            prod = np.multiply(w[:, j:j + 1], r, dtype=np.float32)
            summed = np.add(acc, prod, dtype=np.float32)
        acc = np.where((ok & seen)[:, None], summed, np.where(ok[:, None], prod, acc))
        seen |= ok
    return _bf16.narrow(acc)
