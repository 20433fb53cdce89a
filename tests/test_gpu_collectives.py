"""GPU parity: every collective through the C ABI against the CPU oracle.

Small and ragged sizes that span several reduce tiles, TMA pieces and copy
chunks; every path (copy engines, TMA bulk copies, fused reduce); in-place
forms; misaligned pointers; guard bands around every buffer.
"""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from oracle import alltoall as o_a2a
from oracle import ring as o_ring
from tests.gpu_util import Guarded, assert_bits_equal, to_device, to_host

pytestmark = pytest.mark.gpu

SIZES = [1, 7, 4099, 70001]
PATHS = ["ce", "tma", "fused"]


def _inputs(dtype, k, n, seed):
    rng = np.random.default_rng(seed)
    if dtype == "float32":
        return [(rng.standard_normal(n) * (2.0 ** rng.integers(-20, 20, n))).astype(np.float32) for _ in range(k)]
    return inputs.rank_inputs(dtype, k, n, workload=7, slot=seed % 50)


def _comm(k, path="auto", **kw):
    return hoc.Comm(k, 0, hoc.Config(path=path, **kw))


@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("k", [1, 2, 3, 4, 8, 9, 12, 16])   # 9, 12: the runtime-k fold with a partial last group
@pytest.mark.parametrize("path,engine", [("ce", "lsu"), ("tma", "lsu"), ("fused", "lsu"), ("fused", "tma"),
                                         ("ce", "tma")])
def test_allreduce_parity(dtype, k, path, engine):
    rng = np.random.default_rng(k * 31 + len(path))
    for n in SIZES:
        xs = _inputs(dtype, k, n, seed=n + k)
        order = list(rng.permutation(k))
        want = o_ring.allreduce(xs, dtype, order)
        with _comm(k, path, chunk_bytes=4096, ring_order=order, reduce_engine=engine) as c:
            send = [Guarded(n, dtype) for _ in range(k)]
            recv = [Guarded(n, dtype) for _ in range(k)]
            for g, x in zip(send, xs):
                g.load(x)
            c.allreduce([g.ptr() for g in send], [g.ptr() for g in recv], n, hoc.__dict__[dtype.upper()])
            torch.cuda.synchronize()
            c.wait()
            for r in range(k):
                recv[r].check()
                send[r].check()
                assert_bits_equal(recv[r].host(), want[r], dtype, f"{path} k={k} n={n} rank {r}")
                assert_bits_equal(send[r].host(), xs[r], dtype, "send buffer modified")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("engine", ["lsu", "tma"])
def test_allreduce_in_place_and_misaligned(path, dtype, engine):
    k, n = 4, 12345
    xs = _inputs(dtype, k, n, seed=5)
    want = o_ring.allreduce(xs, dtype)
    code = hoc.FLOAT32 if dtype == "float32" else hoc.BFLOAT16
    with _comm(k, path, chunk_bytes=8192, reduce_engine=engine) as c:
        bufs = [Guarded(n, dtype) for _ in range(k)]
        for g, x in zip(bufs, xs):
            g.load(x)
        c.allreduce([g.ptr() for g in bufs], [g.ptr() for g in bufs], n, code)
        c.wait()
        for r in range(k):
            bufs[r].check()
            assert_bits_equal(bufs[r].host(), want[r], dtype, f"in place {path} rank {r}")
        # pointers shifted by 1..k elements: scalar paths, same bits
        send = [Guarded(n, dtype, offset_elems=r + 1) for r in range(k)]
        recv = [Guarded(n, dtype, offset_elems=(3 * r) % 5) for r in range(k)]
        for g, x in zip(send, xs):
            g.load(x)
        c.allreduce([g.ptr() for g in send], [g.ptr() for g in recv], n, code)
        c.wait()
        for r in range(k):
            recv[r].check()
            assert_bits_equal(recv[r].host(), want[r], dtype, f"misaligned {path} rank {r}")


@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("k", [1, 3, 8, 16])
@pytest.mark.parametrize("engine,budget", [("lsu", 0), ("tma", 0), ("tma", 3), ("lsu", 5)])
def test_reduce_scatter_parity(dtype, k, engine, budget):
    code = hoc.__dict__[dtype.upper()]
    for rc in (1, 5, 3001, 40000):
        xs = _inputs(dtype, k, k * rc, seed=rc + 3 * k)
        want = o_ring.reduce_scatter(xs, rc, dtype)
        with _comm(k, reduce_engine=engine, reduce_max_sms=budget) as c:
            send = [Guarded(k * rc, dtype) for _ in range(k)]
            recv = [Guarded(rc, dtype) for _ in range(k)]
            for g, x in zip(send, xs):
                g.load(x)
            c.reduce_scatter([g.ptr() for g in send], [g.ptr() for g in recv], rc, code)
            c.wait()
            for r in range(k):
                recv[r].check()
                assert_bits_equal(recv[r].host(), want[r], dtype, f"rs k={k} rc={rc} rank {r}")
            # in place: recv[r] = send[r] + r * rc
            c.reduce_scatter([g.ptr() for g in send],
                             [g.ptr() + r * rc * np.dtype(np.float32 if dtype != "bfloat16" else np.uint16).itemsize
                              for r, g in enumerate(send)], rc, code)
            c.wait()
            for r in range(k):
                got = send[r].host()[r * rc:(r + 1) * rc]
                assert_bits_equal(got, want[r], dtype, f"rs in place k={k} rank {r}")


@pytest.mark.parametrize("path", ["ce", "tma"])
@pytest.mark.parametrize("k", [1, 2, 5, 8, 16])
def test_allgather_parity(path, k):
    for sc in (1, 13, 50003):
        xs = inputs.rank_inputs("bfloat16", k, sc, workload=8, slot=k)
        want = o_ring.allgather(xs)
        with _comm(k, path, chunk_bytes=4096) as c:
            send = [Guarded(sc, "bfloat16", offset_elems=r % 3) for r in range(k)]
            recv = [Guarded(k * sc, "bfloat16") for _ in range(k)]
            for g, x in zip(send, xs):
                g.load(x)
            c.allgather([g.ptr() for g in send], [g.ptr() for g in recv], sc, hoc.BFLOAT16)
            c.wait()
            for r in range(k):
                recv[r].check()
                assert_bits_equal(recv[r].host(), want[r], "bfloat16", f"ag {path} k={k} sc={sc} rank {r}")
            st = c.last_stats()
            if path == "ce":
                assert st["kernels"] == 0 and st["sms_used"] == 0
            # in place
            full = [Guarded(k * sc, "bfloat16") for _ in range(k)]
            for r in range(k):
                full[r].tensor[r * sc:(r + 1) * sc].copy_(to_device(xs[r], "bfloat16"))
            c.allgather([g.ptr() + r * sc * 2 for r, g in enumerate(full)], [g.ptr() for g in full], sc, hoc.BFLOAT16)
            c.wait()
            for r in range(k):
                full[r].check()
                assert_bits_equal(full[r].host(), want[r], "bfloat16", f"ag in place {path} rank {r}")


@pytest.mark.parametrize("k", [3, 8, 16])
def test_tma_broadcast_with_mixed_destination_alignment(k):
    # The TMA path loads each source block once and stores it to every
    # destination; destinations in another 16-byte alignment class than the
    # first one get a job of their own.  Receive buffers shifted by 0..7 bf16
    # elements per rank put a block's destinations in several classes.
    for sc in (8, 4099, 300_001):
        xs = inputs.rank_inputs("bfloat16", k, sc, workload=8, slot=20 + k)
        want = o_ring.allgather(xs)
        with _comm(k, "tma", chunk_bytes=1 << 16) as c:
            send = [Guarded(sc, "bfloat16", offset_elems=(5 * r) % 8) for r in range(k)]
            recv = [Guarded(k * sc, "bfloat16", offset_elems=(3 * r) % 8) for r in range(k)]
            for g, x in zip(send, xs):
                g.load(x)
            c.allgather([g.ptr() for g in send], [g.ptr() for g in recv], sc, hoc.BFLOAT16)
            c.wait()
            for r in range(k):
                recv[r].check()
                assert_bits_equal(recv[r].host(), want[r], "bfloat16", f"ag tma mixed k={k} sc={sc} rank {r}")
            # every block is read once (whatever the alignment): the schedule reads kS and writes k*kS
            st = c.last_stats()
            assert st["bytes_exec"] == (k * sc + k * k * sc) * 2


@pytest.mark.parametrize("path", ["ce", "tma"])
@pytest.mark.parametrize("interleave", [True, False])
@pytest.mark.parametrize("stage_sync", [True, False])
def test_alltoallv_parity(path, interleave, stage_sync):
    rng = np.random.default_rng(11)
    for k in (1, 2, 5, 8, 16):
        counts = rng.integers(0, 3000, size=(k, k))
        counts[0, :] = 0 if k > 1 else counts[0, :]
        sends = [rng.integers(0, 1 << 16, size=int(counts[s].sum())).astype(np.uint16) for s in range(k)]
        want = o_a2a.alltoallv(sends, counts)
        lens = o_a2a.recv_lengths(counts)
        with _comm(k, path, chunk_bytes=1024, a2a_interleave=interleave, a2a_stage_sync=stage_sync) as c:
            sb = [Guarded(max(1, len(x)), "bfloat16") for x in sends]
            rb = [Guarded(max(1, n), "bfloat16") for n in lens]
            for g, x in zip(sb, sends):
                if len(x):
                    g.tensor[: len(x)].copy_(to_device(x, "bfloat16"))
            c.alltoall([g.ptr() for g in sb], [g.ptr() for g in rb], sendcounts=counts, dtype=hoc.BFLOAT16)
            c.wait()
            for d in range(k):
                rb[d].check()
                assert_bits_equal(rb[d].host()[: lens[d]], want[d], "bfloat16", f"a2a {path} k={k} dst {d}")


@pytest.mark.parametrize("path", ["ce", "tma"])
def test_alltoall_uniform_involution(path):
    k, cnt = 8, 777
    xs = inputs.rank_inputs("int32", k, k * cnt, workload=8, slot=40)
    with _comm(k, path) as c:
        a = [to_device(x, "int32") for x in xs]
        b = [torch.empty_like(t) for t in a]
        back = [torch.empty_like(t) for t in a]
        c.alltoall(a, b, count=cnt)
        c.alltoall(b, back, count=cnt)
        c.wait()
        want = o_a2a.alltoall_uniform(xs, cnt)
        for r in range(k):
            assert_bits_equal(to_host(b[r], "int32"), want[r], "int32", "uniform a2a")
            assert_bits_equal(to_host(back[r], "int32"), xs[r], "int32", "involution")


@pytest.mark.parametrize("path", ["ce", "tma"])
def test_sendrecv_parity(path):
    with _comm(4, path, chunk_bytes=65536) as c:
        for n in (1, 3, 100003):
            x = inputs.rank_inputs("uint8" if False else "int32", 1, n, workload=8, slot=41)[0].view(np.uint8)
            src = Guarded(len(x), "uint8", offset_elems=3)
            dst = Guarded(len(x), "uint8", offset_elems=5)
            src.load(x)
            c.sendrecv(1, src.ptr(), 2, dst.ptr(), len(x), hoc.UINT8)
            c.wait()
            dst.check()
            assert np.array_equal(dst.host(), x)


@pytest.mark.parametrize("cap", [1, 3, 8])
def test_sm_capped_tma_moves_parity(cap):
    """The TMA copy kernel capped at `cap` CTAs (the 1/2/4/8-SM curves of the sweeps): all-gather,
    all-to-all(v) and send/recv, ragged sizes, misaligned buffers, against the oracle bit for bit."""
    rng = np.random.default_rng(100 + cap)
    for k in (3, 8):
        with _comm(k, "tma", chunk_bytes=1 << 16, copy_max_sms=cap) as c:
            # all-gather: sources and destinations in several 16-byte alignment classes
            for sc in (13, 50_003, 400_001):
                xs = inputs.rank_inputs("bfloat16", k, sc, workload=8, slot=60 + cap)
                want = o_ring.allgather(xs)
                send = [Guarded(sc, "bfloat16", offset_elems=(5 * r + cap) % 8) for r in range(k)]
                recv = [Guarded(k * sc, "bfloat16", offset_elems=(3 * r) % 8) for r in range(k)]
                for g, x in zip(send, xs):
                    g.load(x)
                c.allgather([g.ptr() for g in send], [g.ptr() for g in recv], sc, hoc.BFLOAT16)
                c.wait()
                st = c.last_stats()
                assert st["kernels"] >= 1 and 1 <= st["max_ctas"] <= cap and st["sms_used"] <= cap
                for r in range(k):
                    recv[r].check()
                    assert_bits_equal(recv[r].host(), want[r], "bfloat16", f"capped ag {cap} k={k} sc={sc} rank {r}")
            # all-to-all(v): ragged counts, an empty row and an empty column, misaligned buffers
            counts = rng.integers(0, 40_000, size=(k, k))
            counts[1, :] = 0
            counts[:, 2] = 0
            sends = [rng.integers(0, 1 << 16, size=int(counts[s].sum())).astype(np.uint16) for s in range(k)]
            want = o_a2a.alltoallv(sends, counts)
            lens = o_a2a.recv_lengths(counts)
            sb = [Guarded(max(1, len(x)), "bfloat16", offset_elems=(s + 1) % 8) for s, x in enumerate(sends)]
            rb = [Guarded(max(1, n), "bfloat16", offset_elems=(7 * d) % 8) for d, n in enumerate(lens)]
            for g, x in zip(sb, sends):
                if len(x):
                    g.tensor[: len(x)].copy_(to_device(x, "bfloat16"))
            c.alltoall([g.ptr() for g in sb], [g.ptr() for g in rb], sendcounts=counts, dtype=hoc.BFLOAT16)
            c.wait()
            assert 1 <= c.last_stats()["max_ctas"] <= cap
            for d in range(k):
                rb[d].check()
                assert_bits_equal(rb[d].host()[: lens[d]], want[d], "bfloat16", f"capped a2a {cap} k={k} dst {d}")
            # send/recv: odd byte counts, source and destination misaligned differently
            for n in (1, 4097, 3_000_017):
                x = rng.integers(0, 256, size=n).astype(np.uint8)
                src = Guarded(n, "uint8", offset_elems=3)
                dst = Guarded(n, "uint8", offset_elems=11)
                src.load(x)
                c.sendrecv(0, src.ptr(), k - 1, dst.ptr(), n, hoc.UINT8)
                c.wait()
                assert 1 <= c.last_stats()["max_ctas"] <= cap
                dst.check()
                src.check()
                assert np.array_equal(dst.host(), x), (cap, k, n)


def test_graph_replay_and_profiling_agree():
    k, n = 8, 1 << 20
    xs = inputs.rank_inputs("bfloat16", k, n, workload=2, slot=60, sigma=1e-3)
    want = o_ring.allreduce(xs, "bfloat16")
    for path in ("ce", "tma", "fused"):
        with _comm(k, path, chunk_bytes=1 << 18) as c:
            send = [to_device(x, "bfloat16") for x in xs]
            recv = [torch.empty_like(t) for t in send]
            for it in range(3):
                for t in recv:
                    t.zero_()
                c.allreduce(send, recv)
                st = c.last_stats()
                # a graph is kept for plans with several streams and >= 8 operations
                graphed = path != "fused" and st["kernels"] + st["copies"] >= 8
                assert st["graph_replayed"] == (1 if it > 0 and graphed else 0), (path, it, st)
                c.wait()
                for r in range(k):
                    assert_bits_equal(to_host(recv[r], "bfloat16"), want[r], "bfloat16", f"{path} iter {it}")
            c.profile_enable(True)
            c.allreduce(send, recv)
            c.wait()
            kind = hoc.KERNEL_FUSED if path == "fused" else hoc.KERNEL_REDUCE
            launches, ms = c.profile_read(kind)
            assert launches >= 1 and ms > 0
            for r in range(k):
                assert_bits_equal(to_host(recv[r], "bfloat16"), want[r], "bfloat16", f"{path} profiled")


def test_user_graph_capture():
    k, n = 4, 50000
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=61)
    want = o_ring.allreduce(xs, "float32")
    with _comm(k, "ce", chunk_bytes=16384) as c:
        send = [to_device(x, "float32") for x in xs]
        recv = [torch.empty_like(t) for t in send]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            c.allreduce(send, recv)  # warm the plan cache outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            c.allreduce(send, recv, stream=s)
        for t in recv:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for r in range(k):
            assert_bits_equal(to_host(recv[r], "float32"), want[r], "float32", "captured")


def test_stream_ordering_against_producer_and_consumer():
    """Work before the call on the caller's stream is seen; work after sees the result."""
    k, n = 8, 1 << 22
    with _comm(k, "ce", chunk_bytes=1 << 20) as c:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            send = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(k)]
            recv = [torch.zeros(n, dtype=torch.int32, device="cuda") for _ in range(k)]
            for r in range(k):
                hoc.probe_launch(hoc.sm_count() * 4, 256, 20000, stream=s)  # delay the producer
                send[r].fill_(r + 1)
            c.allreduce(send, recv, stream=s)
            out = torch.stack([t.sum() for t in recv])
        torch.cuda.synchronize()
        assert out.tolist() == [n * k * (k + 1) // 2] * k


def test_errors_are_codes():
    with _comm(2) as c:
        a = torch.zeros(16, dtype=torch.float32, device="cuda")
        b = torch.zeros(16, dtype=torch.float32, device="cuda")
        with pytest.raises(hoc.HocError) as e:
            c.allreduce([a, a], [b, b])          # two ranks share a recv buffer
        assert e.value.code == hoc.ERR_INVALID_ARG
        with pytest.raises(hoc.HocError) as e:
            c.allreduce([a, b], [a.data_ptr() + 2, b.data_ptr()], 4, hoc.FLOAT32)  # misaligned fp32
        assert e.value.code == hoc.ERR_INVALID_ARG
        with pytest.raises(hoc.HocError) as e:
            c.allreduce([a, b], [a, b], 16, hoc.UINT8)
        assert e.value.code == hoc.ERR_UNSUPPORTED
        c.allreduce([a, b], [a, b], 0, hoc.FLOAT32)   # count 0 is a no-op
    with pytest.raises(hoc.HocError) as e:
        hoc.Comm(0)
    assert e.value.code == hoc.ERR_INVALID_ARG
    with pytest.raises(hoc.HocError) as e:
        hoc.Comm(3, 0, hoc.Config(ring_order=[0, 0, 1]))
    assert e.value.code == hoc.ERR_INVALID_ARG


def test_graph_cache_eviction_keeps_results_right():
    """More distinct buffer sets than the graph cache holds (64): evicted graphs are rebuilt."""
    k, n = 4, 20000
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=62)
    want = o_ring.allreduce(xs, "float32")
    with _comm(k, "ce", chunk_bytes=4096) as c:
        sets = []
        for i in range(70):
            send = [to_device(x, "float32") for x in xs]
            recv = [torch.empty_like(t) for t in send]
            sets.append((send, recv))
            c.allreduce(send, recv)
        for send, recv in sets[:3] + sets[-3:]:     # the oldest were evicted, the newest replay
            for t in recv:
                t.zero_()
            c.allreduce(send, recv)
        c.wait()
        for send, recv in sets:
            for r in range(k):
                assert_bits_equal(to_host(recv[r], "float32"), want[r], "float32", "after eviction")


def test_debug_mode_syncs_and_checks(monkeypatch):
    monkeypatch.setenv("HOC_DEBUG", "1")
    k, n = 3, 9999
    xs = inputs.rank_inputs("bfloat16", k, n, workload=7, slot=63)
    want = o_ring.allreduce(xs, "bfloat16")
    for path in ("ce", "tma", "fused"):
        with _comm(k, path, chunk_bytes=2048) as c:
            send = [to_device(x, "bfloat16") for x in xs]
            recv = [torch.empty_like(t) for t in send]
            c.allreduce(send, recv)
            assert c.last_stats()["graph_replayed"] == 0          # debug mode issues directly
            c.wait()
            for r in range(k):
                assert_bits_equal(to_host(recv[r], "bfloat16"), want[r], "bfloat16", f"debug {path}")


def test_two_host_threads_share_a_communicator():
    import threading

    k, n = 4, 100000
    xs = inputs.rank_inputs("int32", k, n, workload=7, slot=64)
    want = o_ring.allreduce(xs, "int32")
    errors = []
    with _comm(k, "ce", chunk_bytes=65536) as c:
        def worker(seed):
            try:
                s = torch.cuda.Stream()
                with torch.cuda.stream(s):
                    send = [to_device(x, "int32") for x in xs]
                    recv = [torch.empty_like(t) for t in send]
                for _ in range(10):
                    c.allreduce(send, recv, stream=s)
                s.synchronize()
                for r in range(k):
                    assert np.array_equal(to_host(recv[r], "int32"), want[r])
            except Exception as e:  # pragma: no cover - reported below
                errors.append(e)
        th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
        for t in th:
            t.start()
        for t in th:
            t.join()
    assert not errors, errors


@pytest.mark.parametrize("path", ["ce", "tma"])
def test_sendrecv_async_completes_by_event(path):
    # The copy waits for the work before the call on the sender's stream and
    # completes `done`; a consumer on another stream waits on `done` alone.
    k, n = 4, (96 << 20) // 2 + 77                      # above 64 MiB: chunks striped over the copy queues
    xs = inputs.rank_inputs("bfloat16", k, n, workload=9, slot=3)
    with _comm(k, path) as c:
        prod, cons = torch.cuda.Stream(), torch.cuda.Stream()
        src = torch.zeros(n, dtype=torch.bfloat16, device="cuda")
        dst = torch.full((n,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        x = to_device(xs[1], "bfloat16")
        with torch.cuda.stream(prod):
            src.copy_(x)                                    # the producer writes the message ...
        done = c.sendrecv_async(1, src, 2, dst, stream=prod)   # ... which the copy waits for
        out = torch.empty_like(dst)
        cons.wait_event(done)
        with torch.cuda.stream(cons):
            out.copy_(dst)                                  # the consumer sees the message
        torch.cuda.synchronize()
        assert_bits_equal(to_host(out, "bfloat16"), xs[1], "bfloat16", f"sendrecv_async {path}")
        # nothing to move: the event still completes
        e = c.sendrecv_async(0, src[:0], 1, dst[:0], stream=prod)
        e.synchronize()


def test_captured_multiwave_reduce_scatters():
    # Whole-GPU reduce-scatters large enough for a multi-wave grid launch with
    # programmatic dependent launch; two of them captured back to back into a
    # CUDA graph keep their order and bits.
    k, rc = 8, 1_638_400
    xs = [inputs.rank_inputs("bfloat16", k, k * rc, workload=3, slot=s) for s in range(2)]
    want = [o_ring.reduce_scatter(x, rc, "bfloat16") for x in xs]
    with _comm(k, "auto") as c:
        send = [[to_device(x, "bfloat16") for x in xs[s]] for s in range(2)]
        recv = [[torch.empty(rc, dtype=torch.bfloat16, device="cuda") for _ in range(k)] for _ in range(2)]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for j in range(2):
                c.reduce_scatter(send[j], recv[j], rc, stream=s)   # plans and occupancy outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for j in range(2):
                c.reduce_scatter(send[j], recv[j], rc, stream=s)
        for j in range(2):
            for t in recv[j]:
                t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for j in range(2):
            for r in range(k):
                assert_bits_equal(to_host(recv[j][r], "bfloat16"), want[j][r], "bfloat16", f"captured rs {j} rank {r}")


@pytest.mark.parametrize("path,engine", [("ce", "lsu"), ("tma", "lsu"), ("fused", "lsu"), ("fused", "tma")])
def test_ring_golden_cases(path, engine):
    """The hand-derived order- and rounding-sensitive cases straight from the golden file (no oracle)."""
    from tests import pins
    torch_dt = {"float32": torch.float32, "int32": torch.int32, "bfloat16": torch.bfloat16}
    view_dt = {"float32": torch.int32, "int32": torch.int32, "bfloat16": torch.int16}
    for c in pins.load_ring_cases():
        k, dt = c["k"], c["dtype"]
        bits_in = [np.asarray(x).view(np.uint32 if dt != "bfloat16" else np.uint16) for x in c["xs"]]
        send = [torch.from_numpy(np.ascontiguousarray(x).view(np.int32 if dt != "bfloat16" else np.int16).copy())
                .cuda().view(torch_dt[dt]) for x in bits_in]
        recv = [torch.zeros_like(t) for t in send]
        with _comm(k, path, ring_order=c["order"], reduce_engine=engine) as comm:
            comm.allreduce(send, recv)
            comm.wait()
        want = c["y"].astype(np.int64)
        for r in range(k):
            got = recv[r].view(view_dt[dt]).cpu().numpy().astype(np.int64) & (0xFFFFFFFF if dt != "bfloat16" else 0xFFFF)
            if dt == "bfloat16":  # a NaN result is compared by class, its payload is free
                nan_w = ((want & 0x7F80) == 0x7F80) & ((want & 0x7F) != 0)
                nan_g = ((got & 0x7F80) == 0x7F80) & ((got & 0x7F) != 0)
                assert np.array_equal(nan_w, nan_g), (c["name"], path)
                assert np.array_equal(got[~nan_w], want[~nan_w]), (c["name"], path, [hex(v) for v in got])
            else:
                assert np.array_equal(got, want), (c["name"], path, [hex(v) for v in got])


@pytest.mark.parametrize("path", ["ce", "tma"])
def test_alltoallv_explicit_displacements(path):
    """Segments placed by explicit displacements: reversed order and gaps on both sides; the gaps of the
    receive buffers keep their fill."""
    from tests.gpu_util import SENTINEL
    rng = np.random.default_rng(12)
    fill = SENTINEL | (SENTINEL << 8)                     # a bf16 element of fill bytes
    for k in (3, 8):
        counts = rng.integers(0, 2000, size=(k, k))
        counts[k - 1, 0] = 0
        sd = np.zeros((k, k), dtype=np.int64)
        rd = np.zeros((k, k), dtype=np.int64)
        for s in range(k):                                # send: destinations in reverse order, gaps of 5
            at = 7
            for d in reversed(range(k)):
                sd[s][d] = at
                at += counts[s][d] + 5
        for d in range(k):                                # receive: sources in reverse order, gaps of 3
            at = 3
            for s in reversed(range(k)):
                rd[d][s] = at
                at += counts[s][d] + 3
        send_len = [int(max(sd[s][d] + counts[s][d] for d in range(k))) for s in range(k)]
        recv_len = [int(max(rd[d][s] + counts[s][d] for s in range(k))) for d in range(k)]
        sends = [rng.integers(0, 1 << 16, size=send_len[s]).astype(np.uint16) for s in range(k)]
        want = o_a2a.alltoallv(sends, counts, sd, rd, recv_len, fill=fill)
        with _comm(k, path, chunk_bytes=1024) as c:
            sb = [Guarded(n, "bfloat16") for n in send_len]
            rb = [Guarded(n, "bfloat16") for n in recv_len]
            for g, x in zip(sb, sends):
                g.load(x)
            c.alltoall([g.ptr() for g in sb], [g.ptr() for g in rb], sendcounts=counts, sdispls=sd, rdispls=rd,
                       dtype=hoc.BFLOAT16)
            c.wait()
            for d in range(k):
                rb[d].check()
                assert_bits_equal(rb[d].host(), want[d], "bfloat16", f"a2a displs {path} k={k} dst {d}")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
@pytest.mark.parametrize("engine,budget", [("lsu", 0), ("tma", 0), ("lsu", 4)])
def test_reduce_scatter_with_a_permuted_ring(dtype, engine, budget):
    """Block r folds from succ(r) around a non-identity ring, as in the allreduce."""
    code = hoc.__dict__[dtype.upper()]
    rng = np.random.default_rng(21)
    for k in (4, 8):
        # k = 4: the reversed ring (with k = 3 every ring gives the same bits: (x_a + x_b) + x_r)
        order = [0, 3, 2, 1] if k == 4 else [int(v) for v in rng.permutation(k)]
        rc = 4099
        xs = _inputs(dtype, k, k * rc, seed=17 + k)
        want = o_ring.reduce_scatter(xs, rc, dtype, order)
        with _comm(k, ring_order=order, reduce_engine=engine, reduce_max_sms=budget) as c:
            send = [Guarded(k * rc, dtype) for _ in range(k)]
            recv = [Guarded(rc, dtype) for _ in range(k)]
            for g, x in zip(send, xs):
                g.load(x)
            c.reduce_scatter([g.ptr() for g in send], [g.ptr() for g in recv], rc, code)
            c.wait()
            for r in range(k):
                recv[r].check()
                assert_bits_equal(recv[r].host(), want[r], dtype, f"rs ring {order} rank {r}")
