"""Two-domain stage scheduler (HOCCL section 3.4): oracle pins and C++ parity.

CPU only.  The oracle (oracle/topo.py) follows Algorithm 1 step by step; it is
pinned to the worked example the paper prints for the traffic matrix (Eq. 5,
Fig. 6), to the completeness and degree constraints (Eqs. 7 and 8), and to
closed forms of special cases.  The C++ scheduler must then reproduce the
oracle's stages exactly.
"""
import numpy as np
import pytest

from collective_communication_schedules_gb300 import hoc
from oracle import topo

# Fig. 6: GPUs g0, g1 in node 0 and g2, g3 in node 1; symmetric peers 0<->1, 2<->3.
FIG6_NODES = [0, 0, 1, 1]
FIG6_SYM = [1, 0, 3, 2]
# Origin matrix of Fig. 6: row g0 = f1 f2 f3, row g1 = f4 f5 f6, row g2 = f7 f8 f9, row g3 = f10 f11 f12
FIG6_CELLS = {(0, 1): 1, (0, 2): 2, (0, 3): 3, (1, 0): 4, (1, 2): 5, (1, 3): 6,
              (2, 0): 7, (2, 1): 8, (2, 3): 9, (3, 0): 10, (3, 1): 11, (3, 2): 12}


def fig6_matrix():
    """f_i = 2^(i-1): every sum of distinct flows has a unique value."""
    C = [[0] * 4 for _ in range(4)]
    for (u, v), i in FIG6_CELLS.items():
        C[u][v] = 1 << (i - 1)
    return C


def f(*idx):
    return sum(1 << (i - 1) for i in idx)


def test_eq5_worked_example():
    T = topo.traffic_matrix(fig6_matrix(), FIG6_NODES, FIG6_SYM)
    # F1 = T[0,1] = f1 + f2' + f3' + f8'' + f11''
    assert T[0][1] == f(1, 2, 3, 8, 11)
    # the other forwarding cells follow the same rule: (u, sym u) gets u's outgoing and sym u's incoming
    assert T[1][0] == f(4, 5, 6, 7, 10)
    assert T[2][3] == f(9, 7, 8, 6, 3)
    assert T[3][2] == f(12, 10, 11, 5, 2)
    # RDMA cells keep their native flow only
    for (u, v), i in FIG6_CELLS.items():
        if FIG6_NODES[u] != FIG6_NODES[v]:
            assert T[u][v] == f(i)


def test_traffic_matrix_by_flows():
    from tests import pins
    pins.check_traffic_matrix_by_flows(topo.traffic_matrix, np.random.default_rng(11))


def _check_invariants(C, nodes, sym, T, stages):
    G = len(C)
    # Eq. 7: the stages sum to T element-wise
    total = [[sum(S[u][v] for S in stages) for v in range(G)] for u in range(G)]
    assert total == T
    # Eq. 8: at most one outgoing and one incoming RDMA flow per GPU per stage
    for S in stages:
        rdma = [(u, v) for u in range(G) for v in range(G) if nodes[u] != nodes[v] and S[u][v] > 0]
        assert len({u for u, _ in rdma}) == len(rdma) == len({v for _, v in rdma})


def _random_case(rng, G, nodes_n):
    nodes = [u * nodes_n // G for u in range(G)]
    sym = [u ^ 1 for u in range(G)]
    C = [[0 if u == v else int(rng.integers(0, 50)) * int(rng.integers(0, 2)) for v in range(G)] for u in range(G)]
    return C, nodes, sym


def test_oracle_invariants_random():
    rng = np.random.default_rng(0)
    for _ in range(60):
        G = int(rng.choice([4, 8]))
        C, nodes, sym = _random_case(rng, G, int(rng.choice([2, 4])) if G == 8 else 2)
        T, stages, taus = topo.schedule(C, nodes, sym, int(rng.integers(1, 20)), int(rng.integers(1, 20)))
        _check_invariants(C, nodes, sym, T, stages)
        assert len(taus) == len(stages) and all(t > 0 for t in taus)


def test_closed_forms():
    # only native intra-node traffic, a permutation within each node: one stage of f / B_nv
    C = [[0, 7, 0, 0], [7, 0, 0, 0], [0, 0, 0, 7], [0, 0, 7, 0]]
    T, stages, taus = topo.schedule(C, FIG6_NODES, FIG6_SYM, 10, 1)
    assert T == C and len(stages) == 1 and taus == [0.7]
    # one inter-node flow u=0 -> v=2 of size 6: one stage with the flow and both forwarding copies
    C = [[0, 0, 6, 0], [0] * 4, [0] * 4, [0] * 4]
    T, stages, taus = topo.schedule(C, FIG6_NODES, FIG6_SYM, 4, 3)
    assert stages == [[[0, 6, 6, 0], [0] * 4, [0] * 4, [0, 0, 6, 0]]]
    assert taus == [max(6 / 3, 6 / 4)]
    # an inter-node permutation (every GPU sends f to its counterpart): one stage, RDMA-bound when B_rdma is low
    C = [[0, 0, 5, 0], [0, 0, 0, 5], [5, 0, 0, 0], [0, 5, 0, 0]]
    T, stages, taus = topo.schedule(C, FIG6_NODES, FIG6_SYM, 100, 1)
    assert len(stages) == 1 and taus == [5.0]


def test_slack_is_filled_without_lengthening_the_stage():
    # an RDMA-bound stage (slow RDMA) leaves NVLink room for the native flow g0 -> g1
    C = [[0, 40, 10, 0], [0] * 4, [0] * 4, [0] * 4]
    T, stages, taus = topo.schedule(C, FIG6_NODES, FIG6_SYM, 10, 1)
    assert len(stages) == 1
    S = stages[0]
    assert S[0][2] == 10 and S[0][1] == 10 + 40   # the forwarding copy plus all native traffic (cap = 100)
    assert taus == [10.0]


def test_cpp_matches_oracle_exactly():
    rng = np.random.default_rng(1)
    cases = [(fig6_matrix(), FIG6_NODES, FIG6_SYM, 9, 2)]
    for _ in range(80):
        G = int(rng.choice([4, 8, 16]))
        C, nodes, sym = _random_case(rng, G, int(rng.choice([2, 4])) if G > 4 else 2)
        cases.append((C, nodes, sym, int(rng.integers(1, 50)), int(rng.integers(1, 50))))
    for C, nodes, sym, bn, br in cases:
        T, stages, taus = topo.schedule(C, nodes, sym, bn, br)
        T2, stages2, taus2, total2 = hoc.topo_schedule(C, nodes, sym, bn, br)
        assert T2 == T
        assert stages2 == stages
        assert taus2 == taus
        assert total2 == pytest.approx(sum(taus), rel=1e-12)


def test_bad_topology_rejected():
    with pytest.raises(hoc.HocError):
        hoc.topo_schedule([[0, 1], [1, 0]], [0, 1], [1, 0], 1, 1)     # symmetric peer in another node
    with pytest.raises(hoc.HocError):
        hoc.topo_schedule([[1, 0], [0, 0]], [0, 0], [1, 0], 1, 1)     # diagonal traffic
