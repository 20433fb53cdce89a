"""Pins of the EP pack / combine oracle (CPU only)."""
import numpy as np

from collective_communication_schedules_gb300 import inputs
from oracle import bf16, ep


def _brute_pack(x, ids, experts, k):
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


def test_pack_matches_brute_force():
    rng = np.random.default_rng(0)
    for _ in range(20):
        k, per = int(rng.integers(1, 5)), int(rng.integers(1, 4))
        experts, tokens, topk, hidden = k * per, int(rng.integers(1, 12)), int(rng.integers(1, 4)), 3
        ids = rng.integers(-1, experts + 1, size=(tokens, topk))          # includes dropped pairs
        x = rng.integers(0, 1 << 16, size=(tokens, hidden)).astype(np.uint16)
        send, perm, pos_of, counts = ep.pack(x, ids, experts, k)
        bperm, brows, bcounts = _brute_pack(x, ids, experts, k)
        assert list(perm) == bperm
        assert np.array_equal(send, np.array(brows, dtype=np.uint16).reshape(-1, hidden))
        assert list(counts) == bcounts
        for row, p in enumerate(perm):
            assert pos_of[p] == row
        assert all(pos_of[p] == -1 for p in range(tokens * topk) if p not in set(bperm))


def test_pack_agrees_with_the_input_generator_layout():
    w = inputs.EP_DISPATCH
    routing = inputs.ep_routing(2, 64, w["experts"], w["topk"], w["zipf"], seed_base=77)
    x = inputs.normal_bf16(64 * 16, 78).reshape(64, 16)
    for r in range(2):
        send, perm, _, counts = ep.pack(x, routing[r], w["experts"], 2)
        gsend, order, gcounts = inputs.ep_pack(routing[r], x, w["experts"], 2)
        assert np.array_equal(send, gsend)
        assert np.array_equal(counts, gcounts * 16)
        assert np.array_equal(perm, order[:, 0] * w["topk"] + order[:, 1])


def test_combine_matches_scalar_brute_force():
    rng = np.random.default_rng(1)
    tokens, topk, hidden = 7, 3, 5
    ids = rng.integers(0, 4, size=(tokens, topk))
    ids[2, 1] = -1                                              # a dropped pair
    x = bf16.narrow(rng.standard_normal((tokens, hidden)).astype(np.float32))
    wts = rng.random(tokens * topk).astype(np.float32)
    send, perm, pos_of, _ = ep.pack(x, ids, 4, 2)
    y = ep.combine(send, pos_of, wts, topk)
    for t in range(tokens):
        for h in range(hidden):
            acc = None
            for j in range(topk):
                p = pos_of[t * topk + j]
                if p < 0:
                    continue
                r = np.float32(bf16.widen(send[p:p + 1, h])[0])
                prod = np.float32(wts[t * topk + j] * r)
                acc = prod if acc is None else np.float32(acc + prod)
            want = bf16.narrow(np.array([0.0 if acc is None else acc], dtype=np.float32))[0]
            assert y[t, h] == want, (t, h)


def test_combine_topk1_unit_weight_is_identity():
    rng = np.random.default_rng(2)
    x = bf16.narrow(rng.standard_normal((9, 4)).astype(np.float32))
    ids = rng.integers(0, 8, size=(9, 1))
    send, _, pos_of, _ = ep.pack(x, ids, 8, 4)
    assert np.array_equal(ep.combine(send, pos_of, np.ones(9, np.float32), 1), x)
