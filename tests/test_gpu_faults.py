"""Failure detection on the GPU without any GPU fault.

Faults are injected on the host (HOC_FAULT): a dropped or duplicated chunk in
the plan must show up as an oracle mismatch; a stalled completion must end
hoc_wait with HOC_ERR_TIMEOUT; a TMA stall (mbarriers that expect bytes that
never arrive) must end the kernel's bounded waits with a status the host
reads, after which the context keeps working.
"""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from oracle import ring as o_ring
from tests.gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu


def _run_allreduce(path, k=4, n=1 << 16):
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=70)
    want = o_ring.allreduce(xs, "float32")
    with hoc.Comm(k, 0, hoc.Config(path=path, chunk_bytes=1 << 14)) as c:
        send = [to_device(x, "float32") for x in xs]
        recv = [torch.full_like(t, float("nan")) for t in send]
        c.allreduce(send, recv)
        c.wait()
    return [to_host(t, "float32") for t in recv], want


@pytest.mark.parametrize("fault", ["drop_chunk", "dup_chunk"])
@pytest.mark.parametrize("path", ["ce", "tma"])
def test_corrupted_plan_is_caught_by_the_oracle(fault, path, monkeypatch):
    monkeypatch.setenv("HOC_FAULT", fault)
    got, want = _run_allreduce(path)
    assert any(not np.array_equal(g.view(np.uint32), w.view(np.uint32)) for g, w in zip(got, want))
    monkeypatch.delenv("HOC_FAULT")
    got, want = _run_allreduce(path)
    assert all(np.array_equal(g.view(np.uint32), w.view(np.uint32)) for g, w in zip(got, want))


def test_stalled_completion_times_out(monkeypatch):
    monkeypatch.setenv("HOC_FAULT", "proxy_stall")
    with hoc.Comm(2, 0) as c:
        a = [torch.ones(1024, device="cuda") for _ in range(2)]
        b = [torch.empty(2048, device="cuda") for _ in range(2)]
        c.allgather(a, b)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=200)
        assert e.value.code == hoc.ERR_TIMEOUT


def test_tma_bounded_wait_reports_and_context_survives(monkeypatch):
    monkeypatch.setenv("HOC_FAULT", "tma_stall")
    with hoc.Comm(2, 0, hoc.Config(path="tma")) as c:
        a = [torch.ones(1 << 16, device="cuda") for _ in range(2)]
        b = [torch.zeros(1 << 17, device="cuda") for _ in range(2)]
        c.allgather(a, b)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_TIMEOUT
        assert "bounded wait" in str(e.value)
    monkeypatch.delenv("HOC_FAULT")
    with hoc.Comm(2, 0, hoc.Config(path="tma")) as c:
        c.allgather(a, b)
        c.wait()
    torch.cuda.synchronize()
    assert bool((b[0] == 1).all()) and bool((b[1] == 1).all())


def test_tma_fed_reduce_bounded_wait_reports_and_context_survives(monkeypatch):
    """The same injected stall in the TMA-fed reduce: every operand slot's mbarrier expects 16 bytes
    that never arrive, the consumers' and the producer's bounded waits give up, the status reaches
    hoc_wait, and the next reduce-scatter is exact."""
    k, n = 4, 1 << 16
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=71)
    want = o_ring.reduce_scatter(xs, n // k, "float32")
    send = [to_device(x, "float32") for x in xs]
    recv = [torch.full((n // k,), float("nan"), device="cuda") for _ in range(k)]
    monkeypatch.setenv("HOC_FAULT", "tma_stall")
    with hoc.Comm(k, 0, hoc.Config(path="ce", reduce_engine="tma")) as c:
        c.reduce_scatter(send, recv, n // k)
        with pytest.raises(hoc.HocError) as e:
            c.wait(timeout_ms=30000)
        assert e.value.code == hoc.ERR_TIMEOUT
        assert "bounded wait" in str(e.value)
    monkeypatch.delenv("HOC_FAULT")
    with hoc.Comm(k, 0, hoc.Config(path="ce", reduce_engine="tma")) as c:
        c.reduce_scatter(send, recv, n // k)
        c.wait()
    for r in range(k):
        assert np.array_equal(to_host(recv[r], "float32").view(np.uint32), want[r].view(np.uint32)), r
