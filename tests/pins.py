"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``check_*`` takes the oracle function(s) under test as arguments and
raises AssertionError on a mismatch, so the same check runs against the real
oracle (tests/test_oracle_*.py) and against planted mistakes
(tests/test_oracle_mutations.py).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from oracle import exact

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- golden file
def load_ring_cases():
    cases = []
    with open(os.path.join(GOLDEN, "ring_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dtype, k, order, inputs, expected = [p.strip() for p in line.split("|")]
            npdt = {"float32": np.uint32, "int32": np.uint32, "bfloat16": np.uint16}[dtype]
            xs = [np.array([int(v, 16) for v in rank.split(",")], dtype=npdt) for rank in inputs.split(";")]
            if dtype == "float32":
                xs = [x.view(np.float32) for x in xs]
            elif dtype == "int32":
                xs = [x.view(np.int32) for x in xs]
            y = np.array([int(v, 16) for v in expected.split(",")], dtype=npdt)
            cases.append(dict(name=name, dtype=dtype, k=int(k), order=[int(v) for v in order.split(",")],
                              xs=xs, y=y))
    return cases


def bits(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float32 or a.dtype == np.int32:
        return a.view(np.uint32)
    return a


def check_golden(allreduce):
    for c in load_ring_cases():
        outs = allreduce(c["xs"], c["dtype"], c["order"])
        assert len(outs) == c["k"], c["name"]
        for o in outs:
            got = bits(o)
            if c["dtype"] == "bfloat16":
                nan_exp = ((c["y"] & 0x7F80) == 0x7F80) & ((c["y"] & 0x7F) != 0)
                nan_got = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
                assert np.array_equal(nan_exp, nan_got), c["name"]
                assert np.array_equal(got[~nan_exp], c["y"][~nan_exp]), (c["name"], got, c["y"])
            else:
                assert np.array_equal(got, c["y"]), (c["name"], [hex(v) for v in got])


# ------------------------------------------------- literal hop-by-hop ring, exact
def literal_ring_rs_f32(xs: list[np.ndarray], order: list[int]) -> list[np.ndarray]:
    """Ring reduce-scatter run hop by hop with exact rounding of each add.

    Written independently of the oracle: positions on the ring are looked up
    here, the partial of block r starts at the rank after r and moves one rank
    forward per step, and the receiving rank adds its own input.
    """
    k = len(xs)
    n = len(xs[0])
    sizes = [n // k + (1 if r < n % k else 0) for r in range(k)]
    offs = [sum(sizes[:r]) for r in range(k)]
    pos = {rank: i for i, rank in enumerate(order)}
    xb = [x.view(np.uint32) for x in xs]
    out = []
    for r in range(k):
        lo, hi = offs[r], offs[r] + sizes[r]
        start = order[(pos[r] + 1) % k]
        partial = [int(v) for v in xb[start][lo:hi]]
        receiver = start
        for step in range(1, k):
            receiver = order[(pos[r] + 1 + step) % k]
            partial = [exact.round_to_f32_bits(exact.f32_bits_to_fraction(p) + exact.f32_bits_to_fraction(int(v)))
                       for p, v in zip(partial, xb[receiver][lo:hi])]
        assert receiver == r
        out.append(np.array(partial, dtype=np.uint32))
    return out


def check_literal_ring(allreduce, rng, trials=40):
    for _ in range(trials):
        k = int(rng.integers(1, 7))
        n = int(rng.integers(1, 40))
        order = list(rng.permutation(k))
        # values of mixed magnitude so that the association order matters
        xs = [(rng.standard_normal(n) * (2.0 ** rng.integers(-30, 10, n))).astype(np.float32) for _ in range(k)]
        want = np.concatenate(literal_ring_rs_f32(xs, order))
        got = allreduce(xs, "float32", order)
        for g in got:
            assert np.array_equal(g.view(np.uint32), want), (k, n, order)


# ------------------------------------------------------- closed forms / bounds
def check_small_integers(allreduce, rng):
    """Integer inputs with small magnitude sum exactly in any order."""
    from collective_communication_schedules_gb300 import inputs
    for dtype, bound in (("float32", 1 << 10), ("bfloat16", 1 << 5), ("int32", 1 << 20)):
        for k in (1, 2, 3, 5, 8):
            xs = inputs.small_int_inputs(dtype, k, 257, int(rng.integers(1 << 30)), bound)
            if dtype == "bfloat16":
                vals = [(x.astype(np.uint32) << 16).view(np.float32).astype(np.float64) for x in xs]
            else:
                vals = [x.astype(np.float64) for x in xs]
            s = np.sum(vals, axis=0)
            for y in allreduce(xs, dtype, None):
                if dtype == "bfloat16":
                    yv = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                else:
                    yv = y.astype(np.float64)
                assert np.array_equal(yv, s), (dtype, k)


def check_int32_wrap(allreduce, rng):
    for k in (2, 3, 8):
        xs = [rng.integers(-(2 ** 31), 2 ** 31, size=101, dtype=np.int64).astype(np.int32) for _ in range(k)]
        s = np.sum([x.astype(np.int64) for x in xs], axis=0)
        want = ((s + 2 ** 31) % 2 ** 32 - 2 ** 31).astype(np.int32)
        for y in allreduce(xs, "int32", list(rng.permutation(k))):
            assert np.array_equal(y, want)


def check_error_bound(allreduce, normalized_error, xs, dtype, tol):
    ys = allreduce(xs, dtype, None)
    err = normalized_error(ys[0], xs, dtype)
    assert float(err.max()) <= tol, float(err.max())
    return float(err.max())


# ------------------------------------------------------- the tolerance metric
def load_tolerance_cases():
    cases = []
    with open(os.path.join(GOLDEN, "tolerance_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dtype, inputs, y, err = [p.strip() for p in line.split("|")]
            npdt, view = {"float32": (np.uint32, np.float32), "bfloat16": (np.uint16, np.uint16)}[dtype]
            xs = [np.array([int(v, 16) for v in rank.split(",")], dtype=npdt).view(view) for rank in inputs.split(";")]
            yv = np.array([int(v, 16) for v in y.split(",")], dtype=npdt).view(view)
            want = [None if e == "inf" else Fraction(e) for e in err.split(",")]
            cases.append(dict(name=name, dtype=dtype, xs=xs, y=yv, err=want))
    return cases


def check_tolerance_golden(normalized_error):
    """The metric on the hand-derived cases, compared exactly (None = +inf)."""
    for c in load_tolerance_cases():
        got = np.asarray(normalized_error(c["y"], c["xs"], c["dtype"]), dtype=np.float64)
        assert got.shape == (len(c["err"]),), c["name"]
        for i, want in enumerate(c["err"]):
            if want is None:
                assert np.isposinf(got[i]), (c["name"], i, got[i])
            else:
                assert got[i] == float(want), (c["name"], i, got[i], float(want))


def check_k1_k2(allreduce, rng):
    x = rng.standard_normal(33).astype(np.float32)
    assert np.array_equal(allreduce([x], "float32", None)[0].view(np.uint32), x.view(np.uint32))
    a = rng.standard_normal(33).astype(np.float32)
    b = rng.standard_normal(33).astype(np.float32)
    want = (a + b).view(np.uint32)            # one IEEE binary32 add
    for y in allreduce([a, b], "float32", None):
        assert np.array_equal(y.view(np.uint32), want)


# -------------------------------------------------------------------- bf16
def check_bf16_narrow_vs_torch(narrow, rng, n=1 << 20):
    import torch
    u = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    # make sure every tie pattern shows up, with odd and even upper halves
    u[: 1 << 12] = (u[: 1 << 12] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = u.view(np.float32)
    got = narrow(x)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
    nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
    assert np.array_equal(nan_w, nan_g)
    assert np.array_equal(got[~nan_w], want[~nan_w])


def check_bf16_narrow_exact(narrow, rng, n=3000):
    u = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    u[:500] = (u[:500] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)      # ties
    u[500:600] = rng.integers(0, 1 << 23, size=100).astype(np.uint32)     # subnormals
    u[600] = 0x7F7FFFFF                                                  # max finite -> inf
    u[601] = 0x7F7F7FFF                                                  # just under the overflow tie
    u[602] = 0x7F7F8000                                                  # overflow tie -> inf
    got = narrow(u.view(np.float32))
    for i, b in enumerate(u):
        v = exact.f32_bits_to_fraction(int(b))
        if v is None:
            continue
        want = exact.round_to_bf16_bits(v)
        if v == 0:
            want |= (int(b) >> 16) & 0x8000
        assert int(got[i]) == want, (hex(int(b)), hex(int(got[i])), hex(want))


# ------------------------------------------------------------------ alltoall
def brute_alltoallv(sends, counts, sdispls, rdispls, recv_lens, fill):
    k = len(sends)
    recvs = [[fill] * recv_lens[d] for d in range(k)]
    for s in range(k):
        for d in range(k):
            for e in range(int(counts[s][d])):
                recvs[d][int(rdispls[d][s]) + e] = sends[s][int(sdispls[s][d]) + e]
    return recvs


def check_alltoallv_brute(alltoallv, rng, trials=30):
    for _ in range(trials):
        k = int(rng.integers(1, 6))
        counts = rng.integers(0, 6, size=(k, k))
        # displacements by explicit running sums (independent of the oracle's helper)
        sd = [[int(sum(counts[s][:d])) for d in range(k)] for s in range(k)]
        rd = [[int(sum(counts[t][d] for t in range(s))) for s in range(k)] for d in range(k)]
        lens = [int(sum(counts[s][d] for s in range(k))) for d in range(k)]
        sends = [rng.integers(0, 1000, size=int(counts[s].sum())).astype(np.int32) for s in range(k)]
        got = alltoallv(sends, counts, np.array(sd), np.array(rd), lens, -1)
        want = brute_alltoallv([list(x) for x in sends], counts, sd, rd, lens, -1)
        for d in range(k):
            assert list(got[d]) == want[d], (k, d)


def check_alltoall_involution(alltoall_uniform, rng):
    for k in (1, 2, 3, 8):
        c = int(rng.integers(0, 9))
        sends = [rng.integers(0, 1 << 16, size=k * c).astype(np.uint16) for _ in range(k)]
        once = alltoall_uniform(sends, c)
        twice = alltoall_uniform(once, c)
        for a, b in zip(sends, twice):
            assert np.array_equal(a, b)
        if k > 1 and c > 0:
            # a transposition, not the identity, unless every block is the same
            assert any(not np.array_equal(a, b) for a, b in zip(sends, once)) or \
                all(np.array_equal(sends[0], s) for s in sends)


def check_alltoallv_inverse(alltoallv, transpose_counts, rng, trials=20):
    for _ in range(trials):
        k = int(rng.integers(1, 9))
        counts = rng.integers(0, 50, size=(k, k))
        sends = [rng.integers(0, 1 << 16, size=int(counts[s].sum())).astype(np.uint16) for s in range(k)]
        mid = alltoallv(sends, counts)
        back = alltoallv(mid, transpose_counts(counts))
        for a, b in zip(sends, back):
            assert np.array_equal(a, b)
        # rows preserved as a multiset
        assert np.array_equal(np.sort(np.concatenate(sends)) if sends else 0,
                              np.sort(np.concatenate(mid)) if mid else 0)
        # receive lengths equal column sums of the send counts
        assert [len(m) for m in mid] == [int(counts[:, d].sum()) for d in range(k)]


def check_shift_stages(shift_stages):
    for k in range(1, 17):
        st = shift_stages(k)
        seen = {}
        for s, stage in enumerate(st):
            outs = [u for u, _ in stage]
            ins = [v for _, v in stage]
            assert len(set(outs)) == len(outs) and len(set(ins)) == len(ins)   # Eq. 8
            for e in stage:
                seen[e] = seen.get(e, 0) + 1
        assert all(seen.get((u, v), 0) == 1 for u in range(k) for v in range(k))   # Eq. 7
        assert len(seen) == k * k


# ------------------------------------------------------------------ pipeline
def check_pipeline_closed_form(simulate, rng):
    for p, m in ((1, 1), (2, 3), (4, 4), (8, 16), (3, 1), (5, 2)):
        keys = rng.integers(1, 1 << 16, size=(p, m, 2)).astype(np.uint16)
        x = [rng.integers(0, 1 << 16, size=17).astype(np.uint16) for _ in range(m)]
        out, trace = simulate(x, keys, p, m)
        for i in range(m):
            key = np.uint16(0)
            for s in range(p):
                key ^= keys[s, i, 0] ^ keys[s, i, 1]
            assert np.array_equal(out[i], x[i] ^ key), (p, m, i)
        assert len(trace) == 2 * p * m


def check_1f1b_shape(one_f_one_b):
    for p in range(1, 9):
        for m in range(1, 17):
            sched = one_f_one_b(p, m)
            assert len(sched) == p
            for s, ops in enumerate(sched):
                f = [mb for kind, mb in ops if kind == "F"]
                b = [mb for kind, mb in ops if kind == "B"]
                assert f == list(range(m)) and b == list(range(m))
                w = min(p - s - 1, m)
                assert [kind for kind, _ in ops[:w]] == ["F"] * w
                # after warm-up no stage holds more than w + 1 forwards without a backward
                inflight, peak = 0, 0
                for kind, _ in ops:
                    inflight += 1 if kind == "F" else -1
                    peak = max(peak, inflight)
                assert peak == min(w + 1, m)


# ------------------------------------------------------------------ EP pack / combine
def _widen_bf16(b) -> np.ndarray:
    """bf16 bit patterns to binary32 (exact: the 16 bits become the high half)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _narrow_bf16_torch(f32) -> np.ndarray:
    """binary32 to bf16 bit patterns by PyTorch's CPU cast (round to nearest even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def brute_ep_pack(x, ids, experts, k):
    """Rows by a literal loop over experts, then tokens, then slots; counts by a per-pair loop."""
    tokens, topk = ids.shape
    perm, rows = [], []
    for e in range(experts):                    # (destination rank, expert) order = expert order
        for t in range(tokens):
            for j in range(topk):
                if ids[t][j] == e:
                    perm.append(t * topk + j)
                    rows.append(x[t])
    counts = [0] * k
    for e in ids.reshape(-1):
        if 0 <= e < experts:
            counts[e // (experts // k)] += x.shape[1]
    return perm, rows, counts


def check_ep_pack_brute(pack, rng, trials=20):
    for _ in range(trials):
        k, per = int(rng.integers(1, 5)), int(rng.integers(1, 4))
        experts, tokens, topk, hidden = k * per, int(rng.integers(1, 12)), int(rng.integers(1, 4)), 3
        ids = rng.integers(-1, experts + 1, size=(tokens, topk))          # includes dropped pairs
        x = rng.integers(0, 1 << 16, size=(tokens, hidden)).astype(np.uint16)
        send, perm, pos_of, counts = pack(x, ids, experts, k)
        bperm, brows, bcounts = brute_ep_pack(x, ids, experts, k)
        assert list(perm) == bperm
        assert np.array_equal(send, np.array(brows, dtype=np.uint16).reshape(-1, hidden))
        assert list(counts) == bcounts
        for row, p in enumerate(perm):
            assert pos_of[p] == row
        assert all(pos_of[p] == -1 for p in range(tokens * topk) if p not in set(bperm))


def check_ep_pack_four_key_sort(pack, x, ids, experts, k):
    """The pack order as a sort on the four keys (destination rank, expert, token, slot) spelled out."""
    tokens, topk = ids.shape
    tok = np.repeat(np.arange(tokens), topk)
    slot = np.tile(np.arange(topk), tokens)
    exp = np.asarray(ids).reshape(-1)
    dst = exp // (experts // k)
    order = np.lexsort((slot, tok, exp, dst))                 # last key is the primary one
    send, perm, _, counts = pack(x, ids, experts, k)
    assert np.array_equal(perm, tok[order] * topk + slot[order])
    assert np.array_equal(send, x[tok[order]])
    assert np.array_equal(counts, np.bincount(dst, minlength=k) * x.shape[1])


def check_ep_combine_scalar(pack, combine, rng):
    """Every output element by a scalar loop of numpy binary32 products and sums, narrowed by PyTorch."""
    tokens, topk, hidden = 7, 3, 5
    ids = rng.integers(0, 4, size=(tokens, topk))
    ids[2, 1] = -1                                              # a dropped pair
    x = _narrow_bf16_torch(rng.standard_normal((tokens, hidden)).astype(np.float32))
    wts = rng.random(tokens * topk).astype(np.float32)
    send, perm, pos_of, _ = pack(x, ids, 4, 2)
    y = combine(send, pos_of, wts, topk)
    for t in range(tokens):
        for h in range(hidden):
            acc = None
            for j in range(topk):
                p = pos_of[t * topk + j]
                if p < 0:
                    continue
                prod = np.float32(wts[t * topk + j] * _widen_bf16(send[p:p + 1, h])[0])
                acc = prod if acc is None else np.float32(acc + prod)
            want = _narrow_bf16_torch(np.array([0.0 if acc is None else acc], dtype=np.float32))[0]
            assert y[t, h] == want, (t, h)


def check_ep_combine_identity(pack, combine, rng):
    """Top-1 with unit weight returns the token rows."""
    x = _narrow_bf16_torch(rng.standard_normal((9, 4)).astype(np.float32))
    ids = rng.integers(0, 8, size=(9, 1))
    send, _, pos_of, _ = pack(x, ids, 8, 4)
    assert np.array_equal(combine(send, pos_of, np.ones(9, np.float32), 1), x)


def load_ep_combine_cases():
    cases = []
    with open(os.path.join(GOLDEN, "ep_combine_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, topk, rows, pos_of, wts, y = [p.strip() for p in line.split("|")]
            cases.append(dict(
                name=name, topk=int(topk),
                rows=np.array([int(v, 16) for v in rows.split(";")], dtype=np.uint16).reshape(-1, 1),
                pos_of=np.array([int(v) for v in pos_of.split(",")], dtype=np.int64),
                weights=np.array([int(v, 16) for v in wts.split(",")], dtype=np.uint32).view(np.float32),
                y=np.array([int(v, 16) for v in y.split(",")], dtype=np.uint16)))
    return cases


def check_ep_combine_golden(combine):
    for c in load_ep_combine_cases():
        got = np.asarray(combine(c["rows"], c["pos_of"], c["weights"], c["topk"])).reshape(-1)
        assert np.array_equal(got, c["y"]), (c["name"], [hex(int(v)) for v in got])


def check_ep_combine_error_bound(pack, combine, rng):
    """|y - s| <= 2^-8 |s| + (topk + 1) 2^-24 sum |w x| against the exact float64 weighted sum s: one
    bf16 rounding of a binary32 fold of topk rounded products (standard error bound of recursive sums)."""
    tokens, topk, hidden = 300, 6, 64
    ids = np.stack([rng.permutation(16)[:topk] for _ in range(tokens)])
    x = _narrow_bf16_torch(rng.standard_normal((tokens, hidden)).astype(np.float32))
    wts = rng.random(tokens * topk).astype(np.float32)
    send, _, pos_of, _ = pack(x, ids, 16, 4)
    y = _widen_bf16(combine(send, pos_of, wts, topk)).astype(np.float64)
    rows = _widen_bf16(send).astype(np.float64)[pos_of.reshape(tokens, topk)]        # [tokens, topk, hidden]
    w = wts.astype(np.float64).reshape(tokens, topk, 1)
    s = (w * rows).sum(axis=1)
    mag = (np.abs(w) * np.abs(rows)).sum(axis=1)
    bound = 2.0 ** -8 * np.abs(s) + (topk + 1) * 2.0 ** -24 * mag * (1 + 2.0 ** -8)
    assert np.all(np.abs(y - s) <= bound + 1e-30)


def random_two_domain_topology(rng):
    """G GPUs in n nodes of equal size (2 or more GPUs each), peers paired within each node."""
    n_nodes = int(rng.choice([2, 3, 4]))
    per = int(rng.choice([2, 4]))
    G = n_nodes * per
    node_of = [u // per for u in range(G)]
    sym = [u ^ 1 for u in range(G)]                 # consecutive pairs, always inside one node
    C = [[0 if u == v else int(rng.integers(0, 40)) * int(rng.integers(0, 2)) for v in range(G)] for u in range(G)]
    return C, node_of, sym


def check_traffic_matrix_by_flows(traffic_matrix, rng, trials=40):
    """Eqs. 2-5 by brute force: route every flow of the origin matrix on its own and add up what each
    GPU pair carries.  A flow inside a node is one NVLink transfer u -> v; a flow between nodes is the
    sender's copy u -> sym[u], the RDMA transfer u -> v (accounted at cell (u, v)) and the receiver's
    copy sym[v] -> v."""
    for _ in range(trials):
        C, node_of, sym = random_two_domain_topology(rng)
        G = len(C)
        load = [[0] * G for _ in range(G)]
        for u in range(G):
            for v in range(G):
                f = C[u][v]
                if u == v or f == 0:
                    continue
                load[u][v] += f
                if node_of[u] != node_of[v]:
                    load[u][sym[u]] += f
                    load[sym[v]][v] += f
        assert traffic_matrix(C, node_of, sym) == load, (C, node_of, sym)
