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


def _traffic_receiver_copy_reversed(C, node_of, sym):
    # the receiver-side forwarding copy counted v -> sym[v] instead of sym[v] -> v
    from oracle import topo
    G = len(C)
    inter, _ = topo.domains(node_of)
    T = [row[:] for row in C]
    for u in range(G):
        for v in range(G):
            if (u, v) in inter and C[u][v]:
                T[u][sym[u]] += C[u][v]
                T[v][sym[v]] += C[u][v]
    return T


def _traffic_no_receiver_copy(C, node_of, sym):
    from oracle import topo
    G = len(C)
    inter, _ = topo.domains(node_of)
    T = [row[:] for row in C]
    for u in range(G):
        T[u][sym[u]] += sum(C[u][v] for v in range(G) if (u, v) in inter)
    return T


@pytest.mark.parametrize("bad", [_traffic_receiver_copy_reversed, _traffic_no_receiver_copy])
def test_topo_traffic_matrix_mistakes_caught(bad):
    assert _fails(pins.check_traffic_matrix_by_flows, bad, np.random.default_rng(11))


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


# ------------------------------------------------------------ EP pack / combine
def _combine_reverse_slots(rows, pos_of, weights, topk):
    from oracle import ep
    pos = np.asarray(pos_of).reshape(-1, topk)[:, ::-1].reshape(-1)
    w = np.asarray(weights, dtype=np.float32).reshape(-1, topk)[:, ::-1].reshape(-1)
    return ep.combine(rows, pos, w, topk)


def _combine_round_every_add(rows, pos_of, weights, topk):
    tokens = len(pos_of) // topk
    w = np.asarray(weights, dtype=np.float32).reshape(tokens, topk)
    pos = np.asarray(pos_of).reshape(tokens, topk)
    acc = np.zeros((tokens, rows.shape[1]), dtype=np.uint16)
    for j in range(topk):
        ok = (pos[:, j] >= 0)[:, None]
        prod = np.multiply(w[:, j:j + 1], bf16.widen(rows[np.where(pos[:, j] >= 0, pos[:, j], 0)]), dtype=np.float32)
        acc = np.where(ok, bf16.narrow(np.add(bf16.widen(acc), prod, dtype=np.float32)), acc)
    return acc


def _combine_ignore_weights(rows, pos_of, weights, topk):
    from oracle import ep
    return ep.combine(rows, pos_of, np.ones(len(pos_of), np.float32), topk)


def _combine_drop_first_slot(rows, pos_of, weights, topk):
    from oracle import ep
    pos = np.asarray(pos_of).reshape(-1, topk).copy()
    pos[:, 0] = -1
    return ep.combine(rows, pos.reshape(-1), weights, topk)


def _combine_unchecked_drop(rows, pos_of, weights, topk):
    # a dropped slot read as row -1 (the last row) instead of skipped
    tokens = len(pos_of) // topk
    w = np.asarray(weights, dtype=np.float32).reshape(tokens, topk)
    pos = np.asarray(pos_of).reshape(tokens, topk)
    acc = np.zeros((tokens, rows.shape[1]), dtype=np.float32)
    for j in range(topk):
        acc = np.add(acc, np.multiply(w[:, j:j + 1], bf16.widen(rows[pos[:, j]]), dtype=np.float32), dtype=np.float32)
    return bf16.narrow(acc)


def _combine_fused_multiply_add(rows, pos_of, weights, topk):
    # each product added unrounded (one rounding per slot, as a fused multiply-add gives)
    tokens = len(pos_of) // topk
    w = np.asarray(weights, dtype=np.float32).reshape(tokens, topk).astype(np.float64)
    pos = np.asarray(pos_of).reshape(tokens, topk)
    acc = np.zeros((tokens, rows.shape[1]), dtype=np.float32)
    seen = np.zeros(tokens, dtype=bool)
    for j in range(topk):
        ok = pos[:, j] >= 0
        prod = w[:, j:j + 1] * bf16.widen(rows[np.where(ok, pos[:, j], 0)]).astype(np.float64)   # exact
        summed = (acc.astype(np.float64) + prod).astype(np.float32)
        acc = np.where((ok & seen)[:, None], summed, np.where(ok[:, None], prod.astype(np.float32), acc))
        seen |= ok
    return bf16.narrow(acc)


@pytest.mark.parametrize("bad", [_combine_reverse_slots, _combine_round_every_add, _combine_ignore_weights,
                                 _combine_drop_first_slot, _combine_unchecked_drop, _combine_fused_multiply_add])
def test_ep_combine_mistakes_caught(bad):
    from oracle import ep
    assert (_fails(pins.check_ep_combine_golden, bad)
            or _fails(pins.check_ep_combine_scalar, ep.pack, bad, np.random.default_rng(7))
            or _fails(pins.check_ep_combine_identity, ep.pack, bad, np.random.default_rng(8))
            or _fails(pins.check_ep_combine_error_bound, ep.pack, bad, np.random.default_rng(10)))


def _pack_tokens_reversed(x, ids, experts, k):
    # unstable within an expert: later tokens first
    from oracle import ep
    tokens, topk = ids.shape
    flat = np.asarray(ids).reshape(-1)
    valid = np.nonzero((flat >= 0) & (flat < experts))[0][::-1]
    perm = valid[np.argsort(flat[valid], kind="stable")].astype(np.int64)
    pos_of = np.full(tokens * topk, -1, dtype=np.int64)
    pos_of[perm] = np.arange(len(perm))
    counts = np.bincount(flat[perm] // (experts // k), minlength=k).astype(np.int64) * x.shape[1]
    return np.ascontiguousarray(x[perm // topk]), perm, pos_of, counts


def _pack_clip_instead_of_drop(x, ids, experts, k):
    from oracle import ep
    return ep.pack(x, np.clip(ids, 0, experts - 1), experts, k)


def _pack_round_robin_ranks(x, ids, experts, k):
    from oracle import ep
    send, perm, pos_of, _ = ep.pack(x, ids, experts, k)
    flat = np.asarray(ids).reshape(-1)
    counts = np.bincount(flat[perm] % k, minlength=k).astype(np.int64) * x.shape[1]   # expert e on rank e % k
    return send, perm, pos_of, counts


@pytest.mark.parametrize("bad", [_pack_tokens_reversed, _pack_clip_instead_of_drop, _pack_round_robin_ranks])
def test_ep_pack_mistakes_caught(bad):
    assert _fails(pins.check_ep_pack_brute, bad, np.random.default_rng(9))


# ------------------------------------------------------------ tolerance metric
def _error_with(num=None, den=None, widen=None, zero=None):
    """normalized_error with one part replaced: numerator, denominator, operand widening or zero rule."""
    def normalized_error(y, xs, dtype):
        wid = widen or (lambda a: ring._widen(a, dtype).astype(np.float64))
        s = sum(wid(x) for x in xs)
        d = den(xs, wid) if den else sum(np.abs(wid(x)) for x in xs)
        yv = wid(y)
        e = num(yv, s) if num else np.abs(yv - s)
        out = np.zeros(len(yv))
        nz = d > 0
        out[nz] = e[nz] / d[nz]
        out[~nz] = zero(yv[~nz]) if zero else np.where(yv[~nz] == 0, 0.0, np.inf)
        return out
    return normalized_error


@pytest.mark.parametrize("bad", [
    _error_with(den=lambda xs, wid: np.abs(sum(wid(x) for x in xs))),            # |s| instead of sum |x|
    _error_with(num=lambda yv, s: np.abs(yv - yv)),                               # y compared with itself
    _error_with(den=lambda xs, wid: sum(wid(x) for x in xs)),                     # the absolute value dropped
    _error_with(num=lambda yv, s: np.abs(yv + s)),                                # sign slip in the numerator
    _error_with(widen=lambda a: np.asarray(a).astype(np.float64)),                # bf16 bit patterns read as integers
    _error_with(widen=lambda a: ring._widen(a, "float32" if np.asarray(a).dtype == np.float32 else "bfloat16")
                .astype(np.float32)),                                             # sums in float32, not float64
    _error_with(zero=lambda yv: np.where(yv == 0, np.inf, 0.0)),                  # zero-denominator rule inverted
])
def test_tolerance_metric_mistakes_caught(bad):
    assert _fails(pins.check_tolerance_golden, bad)
