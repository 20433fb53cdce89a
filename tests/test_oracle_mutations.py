"""Planted mistakes in the oracle must fail at least one pin (CPU only).

Each mutant is a copy of one oracle function with one plausible slip (a wrong
direction, a dropped term, a wrong rounding rule, a transposed operand); the
pins are the same checks the real oracle passes.
"""
import numpy as np
import pytest

from oracle import alltoall, bf16, pipeline, ring
from tests import pins


def _allreduce_with(seq_fn=None, fold_fn=None):
    def allreduce(xs, dtype, order=None):
        k = len(xs)
        order = ring.check_order(order, k)
        n = len(xs[0])
        sizes, offs = ring.block_partition(n, k)
        y = np.empty(n, dtype=np.asarray(xs[0]).dtype)
        for r in range(k):
            seq = (seq_fn or ring.operand_sequence)(r, order)
            lo, hi = offs[r], offs[r] + sizes[r]
            y[lo:hi] = (fold_fn or ring.fold)([xs[j][lo:hi] for j in seq], dtype)
        return [y.copy() for _ in range(k)]
    return allreduce


def _reverse_direction(r, order):
    k = len(order)
    pos = order.index(r)
    return [order[(pos - j) % k] for j in range(1, k + 1)]


def _rank0_first(r, order):
    return list(range(len(order)))


def _ignore_order(r, order):
    return ring.operand_sequence(r, list(range(len(order))))


def _drop_last(operands, dtype):
    return ring.fold(operands[:-1] if len(operands) > 1 else operands, dtype)


def _round_every_hop_bf16(operands, dtype):
    if dtype != "bfloat16":
        return ring.fold(operands, dtype)
    acc = operands[0]
    for v in operands[1:]:
        acc = bf16.narrow(bf16.widen(acc) + bf16.widen(v))
    return acc


def _narrow_ties_away(x):
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x8000)) >> np.uint32(16)).astype(np.uint16)


def _narrow_truncate(x):
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _fails(fn, *args):
    try:
        fn(*args)
    except (AssertionError, ValueError, IndexError):
        return True
    return False


@pytest.mark.parametrize("seq_fn", [_reverse_direction, _rank0_first, _ignore_order])
def test_wrong_ring_order_caught(seq_fn):
    bad = _allreduce_with(seq_fn=seq_fn)
    rng = np.random.default_rng(0)
    assert _fails(pins.check_golden, bad) or _fails(pins.check_literal_ring, bad, rng)


def test_dropped_term_caught():
    bad = _allreduce_with(fold_fn=_drop_last)
    assert _fails(pins.check_small_integers, bad, np.random.default_rng(1))
    assert _fails(pins.check_golden, bad)


def test_rounding_every_hop_caught():
    bad = _allreduce_with(fold_fn=_round_every_hop_bf16)
    assert _fails(pins.check_golden, bad)


@pytest.mark.parametrize("narrow", [_narrow_ties_away, _narrow_truncate])
def test_wrong_bf16_rounding_caught(narrow):
    assert _fails(pins.check_bf16_narrow_vs_torch, narrow, np.random.default_rng(2), 1 << 14)
    assert _fails(pins.check_bf16_narrow_exact, narrow, np.random.default_rng(3), 700)


def test_transposed_alltoall_counts_caught():
    def bad(sends, counts, sd=None, rd=None, lens=None, fill=0):
        c = np.asarray(counts).T
        return alltoall.alltoallv(sends, c, None, None, None, fill)
    assert _fails(pins.check_alltoallv_brute, bad, np.random.default_rng(4))


def test_swapped_displacements_caught():
    def bad(sends, counts, sd=None, rd=None, lens=None, fill=0):
        return alltoall.alltoallv(sends, counts, rd, sd, lens, fill)
    assert _fails(pins.check_alltoallv_brute, bad, np.random.default_rng(5))


def test_bad_stage_decomposition_caught():
    def bad(k):
        return [[(u, (u * s) % k) for u in range(k)] for s in range(k)]
    assert _fails(pins.check_shift_stages, bad)


def test_pipeline_missing_transform_caught():
    def bad(x, keys, p, m):
        keys = keys.copy()
        keys[p - 1, :, 1] = 0          # last stage forgets its backward transform
        return pipeline.simulate(x, keys, p, m)
    assert _fails(pins.check_pipeline_closed_form, bad, np.random.default_rng(6))


# ------------------------------------------------------------ two-domain scheduler
def test_topo_wrong_forwarding_cell_caught():
    from oracle import topo
    from tests import test_topo_sched as tt

    def bad_traffic_matrix(C, node_of, sym):
        G = len(C)
        inter, _ = topo.domains(node_of)
        A = [sum(C[u][v] for v in range(G) if (u, v) in inter) for u in range(G)]
        B = [sum(C[u][v] for u in range(G) if (u, v) in inter) for v in range(G)]
        T = [row[:] for row in C]
        for u in range(G):
            T[u][sym[u]] += A[u] + B[u]          # receiver side on the wrong GPU
        return T

    T = bad_traffic_matrix(tt.fig6_matrix(), tt.FIG6_NODES, tt.FIG6_SYM)
    assert T[0][1] != tt.f(1, 2, 3, 8, 11)


def test_topo_dropped_degree_constraint_caught():
    import numpy as np
    from oracle import topo
    from tests import test_topo_sched as tt

    real = topo.greedy_matching
    try:
        topo.greedy_matching = lambda entries: sorted(entries)          # takes every flow at once
        rng = np.random.default_rng(0)
        caught = False
        for _ in range(20):
            C, nodes, sym = tt._random_case(rng, 8, 2)
            T, stages, _ = topo.schedule(C, nodes, sym, 5, 3)
            caught = caught or _fails(tt._check_invariants, C, nodes, sym, T, stages)
        assert caught
    finally:
        topo.greedy_matching = real
