"""All-to-all(v) and the single-domain stage decomposition.

Semantics (HOCCL section 6.2, "All-to-All"; traffic matrix of section 3.4):
rank s sends cnt[s][d] elements to rank d, taken from its send buffer at
sdispl[s][d]; rank d stores them at rdispl[d][s]:

    recv_d[rdispl[d][s] : rdispl[d][s] + cnt[s][d]] = send_s[sdispl[s][d] : ... + cnt[s][d]]

The default displacements are prefix sums in rank order.  The k x k count
matrix is the origin traffic matrix C of section 3.4 ("Traffic matrix
abstraction"), C[s][d] = flow s -> d.

Stage decomposition (section 3.4, Eq. 6-8) restricted to one domain: the shift
stages T^s = {(u, (u + s) mod k)}, s = 0..k-1, are permutation matchings, so
every rank sends and receives at most one flow per stage (Eq. 8) and the stages
sum to C (Eq. 7).
"""
from __future__ import annotations

import numpy as np


def default_displs(counts: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """sdispl[s][d] = sum_{d' < d} cnt[s][d'];  rdispl[d][s] = sum_{s' < s} cnt[s'][d]."""
    c = np.asarray(counts, dtype=np.int64)
    k = c.shape[0]
    sd = np.zeros((k, k), dtype=np.int64)
    rd = np.zeros((k, k), dtype=np.int64)
    for s in range(k):
        for d in range(1, k):
            sd[s][d] = sd[s][d - 1] + c[s][d - 1]
    for d in range(k):
        for s in range(1, k):
            rd[d][s] = rd[d][s - 1] + c[s - 1][d]
    return sd, rd


def recv_lengths(counts: np.ndarray) -> list[int]:
    c = np.asarray(counts, dtype=np.int64)
    return [int(c[:, d].sum()) for d in range(c.shape[0])]


def alltoallv(sends: list[np.ndarray], counts: np.ndarray, sdispls=None, rdispls=None,
              recv_lens=None, fill=0) -> list[np.ndarray]:
    c = np.asarray(counts, dtype=np.int64)
    k = len(sends)
    if sdispls is None or rdispls is None:
        sd, rd = default_displs(c)
        sdispls = sd if sdispls is None else sdispls
        rdispls = rd if rdispls is None else rdispls
    if recv_lens is None:
        recv_lens = recv_lengths(c)
    dt = np.asarray(sends[0]).dtype
    recvs = [np.full(int(recv_lens[d]), fill, dtype=dt) for d in range(k)]
    for s in range(k):
        for d in range(k):
            n = int(c[s][d])
            a = int(sdispls[s][d])
            b = int(rdispls[d][s])
            recvs[d][b:b + n] = sends[s][a:a + n]
    return recvs


def alltoall_uniform(sends: list[np.ndarray], count: int) -> list[np.ndarray]:
    k = len(sends)
    return alltoallv(sends, np.full((k, k), count, dtype=np.int64))


def transpose_counts(counts: np.ndarray) -> np.ndarray:
    """Counts of the inverse exchange (combine after dispatch)."""
    return np.ascontiguousarray(np.asarray(counts, dtype=np.int64).T)


def shift_stages(k: int) -> list[list[tuple[int, int]]]:
    """Stage s holds the flows (u, (u + s) mod k) for u = 0..k-1."""
    return [[(u, (u + s) % k) for u in range(k)] for s in range(k)]
