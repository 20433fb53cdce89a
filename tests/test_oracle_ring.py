"""Pins of the ring reduce-scatter / allreduce / allgather oracle (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle import ring
from collective_communication_schedules_gb300 import inputs
from tests import pins


def test_block_partition_brute():
    for n in range(0, 40):
        for k in range(1, 9):
            sizes, offs = ring.block_partition(n, k)
            owner = []
            for r in range(k):
                owner += [r] * sizes[r]
            assert len(owner) == n
            assert max(sizes) - min(sizes) <= 1
            assert sorted(sizes, reverse=True) == sizes          # the first n mod k blocks are longer
            assert all(offs[r] == owner.index(r) for r in range(k) if sizes[r])


def test_operand_sequence_ends_with_owner():
    rng = np.random.default_rng(1)
    for k in range(1, 10):
        order = list(rng.permutation(k))
        for r in range(k):
            seq = ring.operand_sequence(r, order)
            assert sorted(seq) == list(range(k)) and seq[-1] == r


def test_golden_cases():
    pins.check_golden(ring.allreduce)


def test_literal_hop_by_hop_ring_exact():
    pins.check_literal_ring(ring.allreduce, np.random.default_rng(7))


def test_k1_identity_k2_single_add():
    pins.check_k1_k2(ring.allreduce, np.random.default_rng(3))


def test_small_integers_exact():
    pins.check_small_integers(ring.allreduce, np.random.default_rng(11))


def test_int32_wraps():
    pins.check_int32_wrap(ring.allreduce, np.random.default_rng(5))


def test_tolerance_metric_golden_cases():
    pins.check_tolerance_golden(ring.normalized_error)


def test_tolerance_metric_refuses_int32():
    # int32 results are compared bit for bit; the metric is defined for floating point only
    with pytest.raises(ValueError):
        ring.normalized_error(np.zeros(2, np.int32), [np.zeros(2, np.int32)] * 2, "int32")


def test_error_bound_fp32_small_workload():
    w = inputs.AR_SMALL
    xs = inputs.rank_inputs("float32", w["k"], w["n"], workload=1)
    e = pins.check_error_bound(ring.allreduce, ring.normalized_error, xs, "float32", ring.TOL["float32"])
    assert e <= (w["k"] - 1) * 2.0 ** -24 * 1.0001


def test_error_bound_bf16():
    xs = inputs.rank_inputs("bfloat16", 8, 1 << 16, workload=2, sigma=1e-3)
    e = pins.check_error_bound(ring.allreduce, ring.normalized_error, xs, "bfloat16", ring.TOL["bfloat16"])
    assert e <= 2.0 ** -8 + 8 * 2.0 ** -24


def test_allreduce_ranks_identical_and_rs_blocks():
    rng = np.random.default_rng(9)
    for dtype in ring.DTYPES:
        for k in (1, 3, 4, 8):
            n = 3 * k + 2
            xs = inputs.rank_inputs(dtype, k, n, workload=9, slot=k)
            ar = ring.allreduce(xs, dtype, list(rng.permutation(k)))
            for y in ar[1:]:
                assert np.array_equal(pins.bits(y), pins.bits(ar[0]))
            rc = 5
            xs2 = inputs.rank_inputs(dtype, k, k * rc, workload=9, slot=10 + k)
            order = list(rng.permutation(k))
            rs = ring.reduce_scatter(xs2, rc, dtype, order)
            ar2 = ring.allreduce(xs2, dtype, order)
            for r in range(k):
                assert np.array_equal(pins.bits(rs[r]), pins.bits(ar2[0][r * rc:(r + 1) * rc]))


def test_allgather_brute():
    rng = np.random.default_rng(4)
    for k in (1, 2, 5):
        xs = [rng.integers(0, 100, size=int(rng.integers(0, 4)) + 3) for _ in range(k)]
        xs = [x[:3] for x in xs]
        out = ring.allgather(xs)
        for r in range(k):
            for s in range(k):
                for e in range(3):
                    assert out[r][3 * s + e] == xs[s][e]


def test_nan_propagates_as_class():
    a = np.array([0x7FA0, 0x3F80], dtype=np.uint16)
    b = np.array([0x3F80, 0xFF81], dtype=np.uint16)
    y = ring.allreduce([a, b], "bfloat16")[0]
    assert oracle.bf16.is_nan_bits(y).all()


def test_bad_order_rejected():
    with pytest.raises(ValueError):
        ring.allreduce([np.zeros(2, np.float32)] * 2, "float32", [0, 0])
