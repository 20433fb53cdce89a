"""The seeded input generators follow the stated recipe (CPU only): shapes of
the five workloads, value distributions, determinism, and the structure of the
expert routing."""
import numpy as np

from collective_communication_schedules_gb300 import inputs


def _widen(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def test_workload_shapes():
    assert inputs.AR_SMALL == dict(k=4, n=1_048_576, dtype="float32", chunks=4)
    assert inputs.AR_LARGE["k"] == 8 and inputs.AR_LARGE["n"] * 2 == 256 << 20      # 256 MiB of bf16 per rank
    rs = inputs.RS_BUCKETS
    assert rs["buckets"] == 268 and rs["bucket_elems"] * 2 == 25 << 20 and rs["bucket_elems"] % rs["k"] == 0
    pp = inputs.PP_STAGES
    assert (pp["p"], pp["microbatches"], pp["seq"] * pp["hidden"] * 2) == (8, 16, 32 << 20)
    ep = inputs.EP_DISPATCH
    assert (ep["k"], ep["tokens"], ep["hidden"], ep["experts"], ep["topk"], ep["zipf"]) == (8, 4096, 2048, 64, 6, 1.1)


def test_value_distributions_and_seeds():
    n = 1 << 18
    f = inputs.rank_inputs("float32", 2, n, workload=1)
    assert all(x.dtype == np.float32 and x.min() >= -1 and x.max() <= 1 for x in f)
    assert abs(f[0].mean()) < 0.01 and abs(f[0].var() - 1 / 3) < 0.01             # U[-1, 1]
    assert np.array_equal(f[1], inputs.uniform_f32(n, 1))                           # workload 1: rank r uses seed r
    b = inputs.rank_inputs("bfloat16", 2, n, workload=2, sigma=1e-3)
    w = _widen(b[0])
    assert abs(w.mean()) < 1e-5 and abs(w.std() / 1e-3 - 1) < 0.01                 # N(0, 1e-3)
    i = inputs.rank_inputs("int32", 8, n, workload=3)
    assert all(x.dtype == np.int32 and x.min() >= -(2 ** 30) and x.max() <= 2 ** 30 for x in i)
    s = np.sum([x.astype(np.int64) for x in i], axis=0)
    assert (np.abs(s) > 2 ** 31 - 1).any()                                          # some 8-rank sums wrap
    assert np.array_equal(inputs.rank_inputs("bfloat16", 2, 99, 2, 5)[1], inputs.rank_inputs("bfloat16", 2, 99, 2, 5)[1])
    assert not np.array_equal(inputs.rank_inputs("bfloat16", 2, 99, 2, 5)[1], inputs.rank_inputs("bfloat16", 2, 99, 2, 6)[1])


def test_expert_routing_structure():
    ep = inputs.EP_DISPATCH
    routing = inputs.ep_routing(2, 2000, ep["experts"], ep["topk"], ep["zipf"])
    p = inputs.zipf_probs(ep["experts"], ep["zipf"])
    assert abs(p.sum() - 1) < 1e-12 and np.all(np.diff(p) < 0)                       # p(e) ~ (e+1)^-1.1, decreasing
    for r in routing:
        assert r.shape == (2000, ep["topk"]) and r.min() >= 0 and r.max() < ep["experts"]
        assert all(len(set(row)) == ep["topk"] for row in r)                        # distinct experts per token
        per_rank = np.bincount(r.reshape(-1) // (ep["experts"] // ep["k"]), minlength=ep["k"])
        assert per_rank[0] == per_rank.max() and per_rank[0] > 2 * per_rank[-1]     # rank 0 hottest
    keys = inputs.pp_keys(8, 16)
    assert keys.shape == (8, 16, 2) and keys.min() >= 1                              # non-zero XOR keys
