"""Stream-memory-operation handshake with the host proxy, on the GPU.

The counts of an all-to-all(v) are computed on the device (as an expert
router would); the caller's stream hands them to the host proxy through the
start / end flags and the proxy moves the data on copy engines.  Checked
against the CPU oracle; the watchdog and error paths must release the stream
(no stream is left waiting on a flag).
"""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from oracle import alltoall as o_a2a
from tests.gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu


def _device_counts(routing_dev, k, experts, hidden):
    """k x k element counts from device-resident routing (the producer kernel)."""
    rows = []
    for r in range(k):
        dst = routing_dev[r].reshape(-1) // (experts // k)
        rows.append(torch.bincount(dst, minlength=k) * hidden)
    return torch.stack(rows).to(torch.int64).contiguous()


def test_device_count_alltoall_matches_oracle():
    k, tokens, hidden, experts, topk = 8, 512, 256, 64, 6
    routing = inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5100)
    counts = np.stack([np.bincount(r.reshape(-1) // (experts // k), minlength=k) for r in routing]) * hidden
    rng = np.random.default_rng(3)
    sends = [rng.integers(0, 1 << 16, size=int(counts[s].sum())).astype(np.uint16) for s in range(k)]
    want = o_a2a.alltoallv(sends, counts)
    lens = o_a2a.recv_lengths(counts)
    # The kernels that run while the stream is held are loaded first: under
    # lazy module loading a first launch can wait for the held stream.  Every
    # operation of the held window below runs once beforehand, on both streams.
    after = torch.zeros(1, device="cuda")
    after += 1
    after.zero_()
    warm = torch.cuda.Stream()
    with torch.cuda.stream(warm):
        after += 1
        after.zero_()
    torch.cuda.synchronize()
    with hoc.Comm(k, 0, hoc.Config(chunk_bytes=1 << 16)) as c:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            after += 1
            rdev = [torch.from_numpy(r).cuda() for r in routing]
            d_counts = _device_counts(rdev, k, experts, hidden)
            sd = [to_device(x, "bfloat16") for x in sends]
            rv = [torch.full((int(lens[d]) + 100,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
                  for d in range(k)]
        c.alltoall_device_counts(sd, rv, d_counts, [t.numel() for t in rv], hoc.BFLOAT16, stream=s)
        after.zero_()
        with torch.cuda.stream(s):
            after += 1                                   # work after the call waits for the moves
        c.wait(s, timeout_ms=30000)
        torch.cuda.synchronize()
        for d in range(k):
            got = to_host(rv[d], "bfloat16")
            assert np.array_equal(got[: lens[d]], want[d]), d
            assert np.all(got[lens[d]:] == 0xFFFF)       # nothing written past the received rows
        st = c.proxy_status()
        assert st["completed"] == 1 and st["released_on_error"] == 0


def test_many_tasks_reuse_slots_and_two_streams():
    k, n = 4, 5000
    rng = np.random.default_rng(9)
    with hoc.Comm(k, 0) as c:
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        for it in range(40):                              # more tasks than proxy slots
            st = streams[it % 2]
            counts = rng.integers(0, n, size=(k, k))
            sends = [rng.integers(0, 1 << 31, size=int(counts[s].sum())).astype(np.int32) for s in range(k)]
            want = o_a2a.alltoallv(sends, counts)
            with torch.cuda.stream(st):
                d_counts = torch.from_numpy(counts.astype(np.int64)).cuda()
                sd = [to_device(x, "int32") if len(x) else torch.zeros(1, dtype=torch.int32, device="cuda") for x in sends]
                rv = [torch.zeros(max(1, int(counts[:, d].sum())), dtype=torch.int32, device="cuda") for d in range(k)]
            c.alltoall_device_counts(sd, rv, d_counts, [t.numel() for t in rv], hoc.INT32, stream=st)
            st.synchronize()
            for d in range(k):
                assert np.array_equal(to_host(rv[d], "int32")[: len(want[d])], want[d]), (it, d)
        assert c.proxy_status()["completed"] == 40


@pytest.mark.parametrize("counts,cap", [
    ([[10, 10], [10, 10]], [5, 20]),                # receiver 0 gets 20 elements into room for 5
    ([[-(1 << 63), 1], [-(1 << 63), 1]], [20, 20]),  # two counts of 2^63 (as uint64): their sum wraps to 0
])
def test_capacity_overflow_releases_the_stream(counts, cap):
    k = 2
    with hoc.Comm(k, 0) as c:
        d_counts = torch.tensor(counts, dtype=torch.int64, device="cuda")
        sd = [torch.ones(20, dtype=torch.int32, device="cuda") for _ in range(k)]
        rv = [torch.zeros(20, dtype=torch.int32, device="cuda") for _ in range(k)]
        c.alltoall_device_counts(sd, rv, d_counts, cap, hoc.INT32)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_INVALID_ARG
        torch.cuda.synchronize()                         # the stream was released
        assert int(rv[0].sum()) == 0 and int(rv[1].sum()) == 0


def test_watchdog_releases_a_stalled_task(monkeypatch):
    monkeypatch.setenv("HOC_FAULT", "proxy_stall")
    k = 2
    with hoc.Comm(k, 0) as c:
        d_counts = torch.tensor([[4, 4], [4, 4]], dtype=torch.int64, device="cuda")
        sd = [torch.ones(8, dtype=torch.int32, device="cuda") for _ in range(k)]
        rv = [torch.zeros(8, dtype=torch.int32, device="cuda") for _ in range(k)]
        c.alltoall_device_counts(sd, rv, d_counts, [8, 8], hoc.INT32)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_TIMEOUT
        torch.cuda.synchronize()
        assert c.proxy_status()["released_on_error"] == 1


def test_callers_on_many_streams():
    # Callers on many streams (more than the hardware work queues): each task
    # is served on the proxy's own streams while its caller is held.
    k, n = 4, 3000
    rng = np.random.default_rng(17)
    streams = [torch.cuda.Stream() for _ in range(24)]
    with hoc.Comm(k, 0) as c:
        for it, st in enumerate(streams):
            counts = rng.integers(0, n, size=(k, k))
            sends = [rng.integers(0, 1 << 31, size=int(counts[s].sum())).astype(np.int32) for s in range(k)]
            want = o_a2a.alltoallv(sends, counts)
            with torch.cuda.stream(st):
                d_counts = torch.from_numpy(counts.astype(np.int64)).cuda()
                sd = [to_device(x, "int32") if len(x) else torch.zeros(1, dtype=torch.int32, device="cuda") for x in sends]
                rv = [torch.zeros(max(1, int(counts[:, d].sum())), dtype=torch.int32, device="cuda") for d in range(k)]
            c.alltoall_device_counts(sd, rv, d_counts, [t.numel() for t in rv], hoc.INT32, stream=st)
            c.wait(st, timeout_ms=30000)
            st.synchronize()
            for d in range(k):
                assert np.array_equal(to_host(rv[d], "int32")[: len(want[d])], want[d]), (it, d)
        st = c.proxy_status()
        assert st["completed"] == len(streams) and st["released_on_error"] == 0


def test_watchdog_releases_while_the_proxy_thread_is_blocked(monkeypatch):
    # Injected on the host: the proxy thread sleeps past the task's deadline
    # (as inside a driver call that waits for the held stream); the watchdog
    # thread, which makes no CUDA call, must release the stream on its own.
    monkeypatch.setenv("HOC_FAULT", "proxy_block")
    k = 2
    with hoc.Comm(k, 0) as c:
        d_counts = torch.tensor([[4, 4], [4, 4]], dtype=torch.int64, device="cuda")
        sd = [torch.ones(8, dtype=torch.int32, device="cuda") for _ in range(k)]
        rv = [torch.zeros(8, dtype=torch.int32, device="cuda") for _ in range(k)]
        torch.cuda.synchronize()
        c.alltoall_device_counts(sd, rv, d_counts, [8, 8], hoc.INT32)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_TIMEOUT
        assert "did not issue the moves" in str(e.value)
        torch.cuda.synchronize()                         # the stream was released
        assert c.proxy_status()["released_on_error"] == 1
        assert int(rv[0].sum()) == 0 and int(rv[1].sum()) == 0   # nothing was moved


def test_send_overflow_releases_the_stream():
    # rank 0's row asks for 20 elements from a send buffer of 15: released before any move
    k = 2
    with hoc.Comm(k, 0) as c:
        d_counts = torch.tensor([[10, 10], [5, 5]], dtype=torch.int64, device="cuda")
        sd = [torch.ones(15, dtype=torch.int32, device="cuda") for _ in range(k)]
        rv = [torch.zeros(20, dtype=torch.int32, device="cuda") for _ in range(k)]
        c.alltoall_device_counts(sd, rv, d_counts, [20, 20], hoc.INT32)     # send capacity: 15 per rank
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_INVALID_ARG and "send buffer" in str(e.value)
        torch.cuda.synchronize()
        assert int(rv[0].sum()) == 0 and int(rv[1].sum()) == 0
        # an explicit send capacity below the tensors' size is what counts
        d_small = torch.tensor([[5, 5], [5, 5]], dtype=torch.int64, device="cuda")
        c.alltoall_device_counts(sd, rv, d_small, [20, 20], hoc.INT32, send_capacity=[9, 15])
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_INVALID_ARG and "send buffer" in str(e.value)
        torch.cuda.synchronize()
        assert int(rv[0].sum()) == 0 and int(rv[1].sum()) == 0


@pytest.mark.parametrize("fault", ["proxy_memop", "proxy_memop_reset"])
def test_failed_stream_operations_release_their_slot(monkeypatch, fault):
    # Injected on the host: the first call's wait for FINISH (or its reset of
    # the end flag) fails to queue.  The call reports HOC_ERR_CUDA and moves
    # nothing; the stream is not held; the slot is freed (or retired, when the
    # end flag would never be reset) and every later call still works.
    monkeypatch.setenv("HOC_FAULT", fault)
    k, n = 2, 64
    rng = np.random.default_rng(23)
    with hoc.Comm(k, 0) as c:
        d_counts = torch.tensor([[n, n], [n, n]], dtype=torch.int64, device="cuda")
        sd = [torch.ones(2 * n, dtype=torch.int32, device="cuda") for _ in range(k)]
        rv = [torch.zeros(2 * n, dtype=torch.int32, device="cuda") for _ in range(k)]
        with pytest.raises(hoc.HocError) as e:
            c.alltoall_device_counts(sd, rv, d_counts, [2 * n, 2 * n], hoc.INT32)
        assert e.value.code == hoc.ERR_CUDA
        torch.cuda.synchronize()                         # the stream passed its flags
        assert int(rv[0].sum()) == 0 and int(rv[1].sum()) == 0
        for it in range(20):                             # more calls than slots: no slot is stuck
            counts = rng.integers(0, 100, size=(k, k))
            sends = [rng.integers(0, 1 << 31, size=int(counts[s].sum())).astype(np.int32) for s in range(k)]
            want = o_a2a.alltoallv(sends, counts)
            dc = torch.from_numpy(counts.astype(np.int64)).cuda()
            sdv = [to_device(x, "int32") if len(x) else torch.zeros(1, dtype=torch.int32, device="cuda") for x in sends]
            rvv = [torch.zeros(max(1, int(counts[:, d].sum())), dtype=torch.int32, device="cuda") for d in range(k)]
            c.alltoall_device_counts(sdv, rvv, dc, [t.numel() for t in rvv], hoc.INT32)
            c.wait(timeout_ms=30000)
            for d in range(k):
                assert np.array_equal(to_host(rvv[d], "int32")[: len(want[d])], want[d]), (it, d)
        st = c.proxy_status()
        assert st["completed"] == 20 and st["released_on_error"] == 0
