"""Pins of the all-to-all(v) oracle and the shift-stage decomposition (CPU only)."""
import numpy as np

from oracle import alltoall
from tests import pins


def test_alltoallv_brute_force():
    pins.check_alltoallv_brute(alltoall.alltoallv, np.random.default_rng(0))


def test_uniform_alltoall_is_involution():
    pins.check_alltoall_involution(alltoall.alltoall_uniform, np.random.default_rng(1))


def test_alltoallv_then_transpose_is_identity():
    pins.check_alltoallv_inverse(alltoall.alltoallv, alltoall.transpose_counts, np.random.default_rng(2))


def test_shift_stages_complete_and_degree_bounded():
    pins.check_shift_stages(alltoall.shift_stages)


def test_default_displs_match_running_sums():
    rng = np.random.default_rng(3)
    c = rng.integers(0, 9, size=(6, 6))
    sd, rd = alltoall.default_displs(c)
    for s in range(6):
        for d in range(6):
            assert sd[s][d] == sum(c[s][:d])
            assert rd[d][s] == sum(c[t][d] for t in range(s))
