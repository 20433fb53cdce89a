"""GPU parity on the five evaluation workloads at their full sizes.

1. ring allreduce, 4 ranks x 1,048,576 fp32 U[-1,1] (seed r), 4 chunks, one copy stream;
2. ring allreduce, 8 ranks x 134,217,728 bf16 N(0, 1e-3), chunk sweep, CE / TMA / fused;
3. DP bucket stream: 8 ranks, 268 x 25 MiB bf16 reduce-scatters back to back with the probe beside;
4. PP send/recv: 8 stages, 16 micro-batches of [1, 4096, 4096] bf16 in 1F1B order;
5. EP dispatch / combine: 8 ranks x 4096 tokens x 2048 bf16, top-6 of 64 experts, Zipf(1.1).

Where the oracle cannot redo the whole output in seconds, the check is on
sampled elements (computed one by one by the oracle) plus properties that hold
at any size (every rank identical, inverse exchange restores the input).
"""
import multiprocessing as mp
from concurrent.futures import ProcessPoolExecutor

import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from collective_communication_schedules_gb300.pipeline import Pipeline1F1B
from oracle import alltoall as o_a2a
from oracle import ep as o_ep
from oracle import pipeline as o_pp
from oracle import ring as o_ring
from tests.gpu_util import assert_bits_equal, to_device, to_host

pytestmark = pytest.mark.gpu


def _pool_map(fn, args):
    with ProcessPoolExecutor(max_workers=8, mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(fn, args))


def _gen_large(r):
    return inputs.normal_bf16(134_217_728, inputs.seed_for(2, 0, r), 1e-3)


def _gen_bucket(args):
    slot, r = args
    return inputs.normal_bf16(13_107_200, inputs.seed_for(3, slot, r), 1e-3)


# ------------------------------------------------------------------ workload 1
@pytest.mark.parametrize("path", ["ce", "tma", "fused"])
@pytest.mark.parametrize("dtype", ["float32", "int32"])
def test_small_allreduce_workload(path, dtype):
    w = inputs.AR_SMALL
    k, n = w["k"], w["n"]
    xs = inputs.rank_inputs(dtype, k, n, workload=1)
    want = o_ring.allreduce(xs, dtype)
    chunk = (n // k) * 4 // w["chunks"]                     # 4 chunks per block
    code = hoc.FLOAT32 if dtype == "float32" else hoc.INT32
    with hoc.Comm(k, 0, hoc.Config(path=path, chunk_bytes=chunk, n_copy_streams=1)) as c:
        send = [to_device(x, dtype) for x in xs]
        recv = [torch.empty_like(t) for t in send]
        c.allreduce(send, recv, n, code)
        c.wait()
        if path != "fused":
            assert c.last_stats()["kernels"] == (w["chunks"] if path == "ce" else 2 * w["chunks"])
        for r in range(k):
            got = to_host(recv[r], dtype)
            assert_bits_equal(got, want[r], dtype, f"workload 1 {path} rank {r}")
        if dtype == "float32":
            err = o_ring.normalized_error(to_host(recv[0], dtype), xs, dtype)
            assert err.max() <= o_ring.TOL["float32"]


# ------------------------------------------------------------------ workload 2
@pytest.fixture(scope="module")
def large_inputs():
    xs = _pool_map(_gen_large, range(8))
    dev = [to_device(x, "bfloat16") for x in xs]
    rng = np.random.default_rng(2024)
    idx = np.sort(rng.choice(134_217_728, size=1 << 20, replace=False))
    blk = 134_217_728 // 8
    owners = idx // blk
    want = np.empty(len(idx), dtype=np.uint16)
    for r in range(8):
        sel = owners == r
        cols = [x[idx[sel]] for x in xs]
        seq = o_ring.operand_sequence(r, list(range(8)))
        want[sel] = o_ring.fold([cols[j] for j in seq], "bfloat16")
    err_ref = o_ring.normalized_error(want, [x[idx] for x in xs], "bfloat16")
    assert err_ref.max() <= o_ring.TOL["bfloat16"]
    return dev, idx, want


@pytest.mark.parametrize("path,chunk_mib,engine", [("fused", 4, "lsu"), ("fused", 4, "tma"), ("ce", 1, "lsu"),
                                                    ("ce", 4, "lsu"), ("ce", 16, "tma"), ("ce", 64, "lsu"),
                                                    ("tma", 4, "lsu"), ("tma", 32, "lsu")])
def test_large_allreduce_workload(large_inputs, path, chunk_mib, engine):
    send, idx, want = large_inputs
    recv = [torch.empty_like(t) for t in send]
    with hoc.Comm(8, 0, hoc.Config(path=path, chunk_bytes=chunk_mib << 20, reduce_engine=engine)) as c:
        c.allreduce(send, recv)
        c.wait()
        st = c.last_stats()
    ti = torch.from_numpy(idx).cuda()
    for r in range(8):
        got = recv[r].view(torch.int16).index_select(0, ti).cpu().numpy().view(np.uint16)
        assert_bits_equal(got, want, "bfloat16", f"workload 2 {path} {chunk_mib} MiB rank {r}")
        if r:
            assert torch.equal(recv[r].view(torch.int16), recv[0].view(torch.int16)), f"rank {r} differs from rank 0"
    if path == "ce":
        assert st["copies"] == 56 * max(1, 32 // min(chunk_mib, 32))


# ------------------------------------------------------------------ workload 3
@pytest.mark.parametrize("budget,engine", [(0, "lsu"), (16, "tma")])
def test_bucket_stream_reduce_scatter_workload(budget, engine):
    w = inputs.RS_BUCKETS
    k, nb, be, pool = w["k"], w["buckets"], w["bucket_elems"], w["pool"]
    rc = be // k
    host = _pool_map(_gen_bucket, [(s, r) for s in range(pool) for r in range(k)])
    pool_in = [[to_device(host[s * k + r], "bfloat16") for r in range(k)] for s in range(pool)]
    expected = []
    for s in range(pool):
        ys = o_ring.reduce_scatter(host[s * k:(s + 1) * k], rc, "bfloat16")
        expected.append([to_device(y, "bfloat16") for y in ys])
    outs = torch.empty((nb, k, rc), dtype=torch.bfloat16, device="cuda")
    sms = hoc.sm_count()
    probe_stream = torch.cuda.Stream()
    coll_stream = torch.cuda.Stream()
    with hoc.Comm(k, 0, hoc.Config(reduce_max_sms=budget, reduce_engine=engine)) as c:
        hoc.probe_launch(64 * sms, 256, 4000, stream=probe_stream)
        for b in range(nb):
            c.reduce_scatter(pool_in[b % pool], [outs[b, r] for r in range(k)], rc, stream=coll_stream)
        torch.cuda.synchronize()
        c.wait()
        assert c.last_stats()["kernels"] == 1
    for b in range(nb):
        for r in range(k):
            assert torch.equal(outs[b, r].view(torch.int16), expected[b % pool][r].view(torch.int16)), (b, r)


# ------------------------------------------------------------------ workload 4
@pytest.mark.parametrize("path", ["ce", "tma"])
@pytest.mark.parametrize("sends", ["pull", "event", "stream"])
def test_pipeline_1f1b_workload(path, sends):
    w = inputs.PP_STAGES
    p, m = w["p"], w["microbatches"]
    elems = w["seq"] * w["hidden"]
    keys = inputs.pp_keys(p, m)
    xs = inputs.pp_activations(m, elems)
    want, _ = o_pp.simulate(xs, keys, p, m)
    sms = hoc.sm_count()
    with hoc.Comm(p, 0, hoc.Config(path=path)) as c:
        pipe = Pipeline1F1B(c, p, m, elems, keys, probe_ctas=2 * sms, probe_iters=2000, sends=sends)
        pipe.load([to_device(x, "bfloat16") for x in xs])
        pipe.issue()
        torch.cuda.synchronize()
        c.wait()
        for i in range(m):
            got = pipe.result(i).cpu().numpy().view(np.uint16)
            assert_bits_equal(got, want[i], "bfloat16", f"pp micro-batch {i}")
        # the issue order is a valid 1F1B execution: per stage it follows the schedule
        per_stage = [[(kind, i) for s2, kind, i in pipe.issue_trace if s2 == s] for s in range(p)]
        assert per_stage == o_pp.one_f_one_b(p, m)


# ------------------------------------------------------------------ workload 5
@pytest.fixture(scope="module")
def ep_data():
    w = inputs.EP_DISPATCH
    routing = inputs.ep_routing(w["k"], w["tokens"], w["experts"], w["topk"], w["zipf"])
    xs = inputs.ep_token_rows(w["k"], w["tokens"], w["hidden"])
    packs = [o_ep.pack(xs[r], routing[r], w["experts"], w["k"]) for r in range(w["k"])]
    sends = [p[0] for p in packs]
    counts = np.stack([p[3] for p in packs]) // w["hidden"]         # rows per (source, destination)
    return w, sends, counts, routing


@pytest.mark.parametrize("path,interleave", [("ce", True), ("ce", False), ("tma", True)])
def test_expert_dispatch_combine_workload(ep_data, path, interleave):
    w, sends, counts, routing = ep_data
    k, h = w["k"], w["hidden"]
    assert counts.sum() == k * w["tokens"] * w["topk"]
    assert counts[:, 0].sum() == counts.sum(axis=0).max()            # rank 0 holds the hottest experts
    flat = [s.reshape(-1) for s in sends]
    ecounts = counts * h
    want = o_a2a.alltoallv(flat, ecounts)
    lens = o_a2a.recv_lengths(ecounts)
    with hoc.Comm(k, 0, hoc.Config(path=path, a2a_interleave=interleave)) as c:
        sd = [to_device(x, "bfloat16") for x in flat]
        rv = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for n in lens]
        back = [torch.empty_like(t) for t in sd]
        c.alltoall(sd, rv, sendcounts=ecounts, dtype=hoc.BFLOAT16)
        c.alltoall(rv, back, sendcounts=o_a2a.transpose_counts(ecounts), dtype=hoc.BFLOAT16)
        c.wait()
        for d in range(k):
            assert_bits_equal(to_host(rv[d], "bfloat16"), want[d], "bfloat16", f"dispatch dst {d}")
        for s in range(k):
            assert torch.equal(back[s].view(torch.int16), sd[s].view(torch.int16)), f"combine src {s}"


@pytest.mark.parametrize("whole_sm", [False, True])
def test_probe_launch_flags(whole_sm):
    """The FMA probe with and without programmatic dependent launch: a train of each runs and
    reports the clock it ran at; a flag bit the call does not know is refused."""
    sms = hoc.sm_count()
    threads = 1024 if whole_sm else 256
    s = torch.cuda.Stream()
    for pdl in (False, True):
        sink = torch.zeros(4, dtype=torch.float32, device="cuda")
        for _ in range(3):
            hoc.probe_launch(sms, threads, 2000, sink=sink, stream=s, whole_sm=whole_sm, pdl=pdl)
        torch.cuda.synchronize()
        cyc, ns = float(sink[0]), float(sink[1])
        assert cyc > 0 and ns > 0 and 500 < 1e3 * cyc / ns < 3000, (pdl, cyc, ns)   # MHz
    assert hoc.lib().hoc_probe_launch(s.cuda_stream, 1, 32, 1, 4, None) == hoc.ERR_INVALID_ARG
