"""Per-stream finish profiling (the tail of a schedule over the copy streams), on the GPU."""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc
from oracle import alltoall as o_a2a
from tests.gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu


def test_stream_finish_times_of_a_multi_stream_alltoall():
    k, n = 8, 1 << 20
    rng = np.random.default_rng(21)
    counts = rng.integers(0, n // k, size=(k, k))
    sends = [rng.integers(0, 1 << 31, size=int(counts[s].sum())).astype(np.int32) for s in range(k)]
    want = o_a2a.alltoallv(sends, counts)
    s = torch.cuda.Stream()
    with hoc.Comm(k, 0, hoc.Config(path="ce", n_copy_streams=4, chunk_bytes=1 << 18)) as c:
        sd = [to_device(x, "int32") for x in sends]
        rv = [torch.zeros(int(counts[:, d].sum()), dtype=torch.int32, device="cuda") for d in range(k)]
        torch.cuda.synchronize()
        c.profile_enable(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        c.alltoall(sd, rv, sendcounts=counts, dtype=hoc.INT32, stream=s)
        e1.record(s)
        fin = c.profile_stream_finish()
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
        assert 2 <= len(fin) <= 4                       # the call forked onto the copy streams
        assert all(0 < v <= total + 0.05 for v in fin)  # each stream ends inside the call
        for d in range(k):
            assert np.array_equal(to_host(rv[d], "int32"), want[d]), d
        # a call on the caller's stream alone reports no copy streams
        a = torch.ones(1024, dtype=torch.int32, device="cuda")
        b = torch.zeros(1024, dtype=torch.int32, device="cuda")
        c.sendrecv(0, a, 1, b, stream=s)
        assert c.profile_stream_finish() == []
        c.profile_enable(False)


def test_timeline_of_a_pipelined_allreduce():
    # Copy-engine allreduce in 4 chunks per block: one reduce step per chunk on
    # the caller's stream, then that chunk's copies on the copy queues, each
    # starting only once its chunk's reduce has ended; results stay exact.
    from oracle import ring as o_ring
    from collective_communication_schedules_gb300 import inputs
    k, n, chunks = 4, 1 << 18, 4
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=62)
    want = o_ring.allreduce(xs, "float32")
    s = torch.cuda.Stream()
    with hoc.Comm(k, 0, hoc.Config(path="ce", n_copy_streams=2, chunk_bytes=(n // k) * 4 // chunks)) as c:
        send = [to_device(x, "float32") for x in xs]
        recv = [torch.empty_like(t) for t in send]
        torch.cuda.synchronize()
        c.profile_enable(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        c.allreduce(send, recv, stream=s)
        e1.record(s)
        tl = c.profile_timeline()
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
        c.profile_enable(False)
        reduces = [t for t in tl if t["kind"] == "reduce"]
        copies = [t for t in tl if t["kind"] == "copy"]
        assert [t["stage"] for t in reduces] == list(range(chunks))
        assert all(t["stream"] == 0 for t in reduces)
        assert {t["stage"] for t in copies} == set(range(chunks)) and all(t["stream"] >= 1 for t in copies)
        for t in tl:
            assert -0.01 <= t["start_ms"] <= t["end_ms"] <= total + 0.05, t
        for t in copies:                                  # a chunk's moves wait for its reduce
            assert t["start_ms"] >= reduces[t["stage"]]["end_ms"] - 1e-3, (t, reduces[t["stage"]])
        for r in range(k):
            assert np.array_equal(to_host(recv[r], "float32").view(np.uint32), want[r].view(np.uint32))


def test_timeline_of_a_captured_call_after_replay():
    # profiled inside the caller's graph capture: the timeline is that of the last replay
    k, n = 4, 1 << 16
    s = torch.cuda.Stream()
    with hoc.Comm(k, 0, hoc.Config(path="ce", n_copy_streams=2, chunk_bytes=(n // k) * 4 // 2)) as c:
        send = [torch.ones(n, device="cuda") for _ in range(k)]
        recv = [torch.zeros(n, device="cuda") for _ in range(k)]
        with torch.cuda.stream(s):
            c.allreduce(send, recv, stream=s)          # plans built outside the capture
        torch.cuda.synchronize()
        c.profile_enable(True)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            c.allreduce(send, recv, stream=s)
        c.profile_enable(False)
        for t in recv:
            t.zero_()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        tl = c.profile_timeline()
        assert {t["kind"] for t in tl} == {"reduce", "copy"}
        assert all(0 <= t["start_ms"] <= t["end_ms"] < 100 for t in tl)
        assert all(bool((r == k).all()) for r in recv)
        launches, ms = c.profile_read(hoc.KERNEL_REDUCE)     # the kernel events of the capture are readable too
        assert launches == 2 and ms > 0
