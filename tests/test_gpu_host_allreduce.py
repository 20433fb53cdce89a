"""AllReduce over host buffers against the oracle, in both modes: direct (one fused launch on host memory the
device addresses) and staged (copy-engine pipeline through device slots)."""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from oracle import ring as o_ring

pytestmark = pytest.mark.gpu


def _host(x, dtype, pinned):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16) if dtype == "bfloat16" else np.ascontiguousarray(x))
    t = t.view(torch.bfloat16) if dtype == "bfloat16" else t
    return t.pin_memory() if pinned else t.clone()


def _bits(t, dtype):
    a = t.view(torch.int16).numpy().view(np.uint16) if dtype == "bfloat16" else t.numpy()
    return a.view(np.uint32) if a.dtype in (np.float32, np.int32) else a


@pytest.mark.parametrize("dtype", ["int32", "float32", "bfloat16"])
@pytest.mark.parametrize("k", [1, 3, 8])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("path", ["auto", "ce"])
def test_host_allreduce_matches_oracle(dtype, k, pinned, path):
    rng = np.random.default_rng(k)
    order = list(rng.permutation(k))
    with hoc.Comm(k, 0, hoc.Config(ring_order=order, path=path)) as c:
        for n in (1, 4099, 5_000_003):                   # several 8 MiB chunks and a ragged tail
            xs = inputs.rank_inputs(dtype, k, n, workload=7, slot=(n + k) % 50)
            want = o_ring.allreduce(xs, dtype, order)
            hs = [_host(x, dtype, pinned) for x in xs]
            hr = [torch.empty_like(t) for t in hs]
            if pinned:
                hr = [t.pin_memory() for t in hr]
            for _ in range(2):                             # second call replays the cached graph
                for t in hr:
                    t.zero_()
                c.allreduce_host(hs, hr)
                c.wait()
                torch.cuda.synchronize()
                st = c.last_stats()
                if path == "ce":
                    assert st["copies"] > 0                # staged through the copy engines
                elif pinned:
                    assert st["path"] == hoc.PATH_FUSED and st["copies"] == 0 and st["kernels"] == 1   # direct
                for r in range(k):
                    w = want[r].view(np.uint32) if want[r].dtype in (np.float32, np.int32) else want[r]
                    got = _bits(hr[r], dtype)
                    if dtype == "bfloat16":
                        nan = ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
                        assert np.array_equal(got[~nan], w[~nan]), (n, r)
                    else:
                        assert np.array_equal(got, w), (n, r)


def test_host_allreduce_in_place():
    k, n = 4, 3_000_001
    xs = inputs.rank_inputs("float32", k, n, workload=7, slot=33)
    want = o_ring.allreduce(xs, "float32")
    hs = [torch.from_numpy(x.copy()).pin_memory() for x in xs]
    with hoc.Comm(k, 0) as c:
        c.allreduce_host(hs, hs)
        c.wait()
    torch.cuda.synchronize()
    for r in range(k):
        assert np.array_equal(hs[r].numpy().view(np.uint32), want[r].view(np.uint32))
