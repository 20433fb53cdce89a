"""The allocation-free TMA moves entry point against the communicator path.

hoc_tma_moves_noalloc exists for callers that cannot call cudaMalloc (for
example a plug-in inside a runtime whose allocator already holds the GPU's
memory).  It must move exactly what hoc_allgather moves on the TMA path, call
after call: the shared scratch array keeps the previous call's contents, so
two calls in a row with different data are compared.  This file is collected
last so a failure here does not hide any other test.
"""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


def _allgather_moves(send, recv, sc_bytes, offset):
    src, dst, nb = [], [], []
    for r in range(len(send)):
        for d in range(len(send)):
            src.append(send[r].data_ptr() + offset)
            dst.append(recv[d].data_ptr() + offset + r * sc_bytes)
            nb.append(sc_bytes)
    return src, dst, nb


@pytest.mark.parametrize("offset", [0, 3])
def test_noalloc_moves_match_allgather_twice(offset):
    k, sc = 4, 300_007                                    # int32 elements per rank
    sc_bytes = sc * 4
    with hoc.Comm(k, 0, hoc.Config(path="tma")) as comm:
        for call in range(2):
            xs = inputs.rank_inputs("int32", k, sc, workload=9, slot=80 + call)
            send = [torch.zeros(sc_bytes + 64, dtype=torch.uint8, device="cuda") for _ in range(k)]
            for r in range(k):
                send[r][offset:offset + sc_bytes].copy_(to_device(xs[r], "int32").view(torch.uint8))
            ref = [torch.zeros(k * sc_bytes + 64, dtype=torch.uint8, device="cuda") for _ in range(k)]
            new = [torch.zeros(k * sc_bytes + 64, dtype=torch.uint8, device="cuda") for _ in range(k)]
            comm.allgather([t.data_ptr() + offset for t in send], [t.data_ptr() + offset for t in ref], sc_bytes,
                           hoc.UINT8)
            comm.wait()
            src, dst, nb = _allgather_moves(send, new, sc_bytes, offset)
            hoc.tma_moves_noalloc(src, dst, nb, wait=True)
            torch.cuda.synchronize()
            for d in range(k):
                assert torch.equal(new[d], ref[d]), f"call {call} rank {d}"
                got = new[d][offset:offset + k * sc_bytes].cpu().numpy().view(np.int32)
                assert np.array_equal(got, np.concatenate(xs)), f"call {call} rank {d} content"


def test_noalloc_rejects_too_many_moves():
    a = torch.zeros(16, dtype=torch.uint8, device="cuda")
    b = torch.zeros(16, dtype=torch.uint8, device="cuda")
    n = hoc.NOALLOC_MAX_MOVES + 1
    with pytest.raises(hoc.HocError) as e:
        hoc.tma_moves_noalloc([a] * n, [b] * n, [16] * n)
    assert e.value.code == hoc.ERR_INVALID_ARG
    assert "192" in str(e.value)


def test_noalloc_allocates_no_device_memory():
    # The entry point's promise: after the first call on the device (which sets
    # it up), calls leave the device's free memory unchanged.
    n = 1 << 22
    a = torch.arange(n, dtype=torch.int32, device="cuda").view(torch.uint8)
    b = torch.zeros_like(a)
    src, dst, nb = [a.data_ptr()], [b.data_ptr()], [a.numel()]
    for _ in range(2):
        hoc.tma_moves_noalloc(src, dst, nb, wait=True)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        hoc.tma_moves_noalloc(src, dst, nb, wait=True)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert torch.equal(a, b)


def test_noalloc_bounded_wait_reports_timeout_then_recovers(monkeypatch):
    # Injected on the host: every mbarrier of the bulk-copy kernel expects 16
    # bytes more than its load brings, so its bounded waits give up (0.1 s) and
    # the status word in the shared scratch array reports it.  The next call
    # clears the array and moves the bytes.
    n = 1 << 20
    a = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    monkeypatch.setenv("HOC_FAULT", "tma_stall")
    with pytest.raises(hoc.HocError) as e:
        hoc.tma_moves_noalloc([a], [b], [n], wait=True)
    assert e.value.code == hoc.ERR_TIMEOUT
    monkeypatch.delenv("HOC_FAULT")
    b.zero_()
    hoc.tma_moves_noalloc([a], [b], [n], wait=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_noalloc_rejects_null_and_huge_moves():
    a = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(hoc.HocError) as e:
        hoc.tma_moves_noalloc([0], [a.data_ptr()], [16])
    assert e.value.code == hoc.ERR_INVALID_ARG and "NULL" in str(e.value)
    with pytest.raises(hoc.HocError) as e:                 # nothing is queued: the size check comes first
        hoc.tma_moves_noalloc([a.data_ptr()], [a.data_ptr() + (1 << 41)], [(1 << 40) + 1])
    assert e.value.code == hoc.ERR_INVALID_ARG and "2^40" in str(e.value)
