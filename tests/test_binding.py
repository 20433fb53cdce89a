"""The binding's argument marshalling, on CPU: every tensor a call hands the
library must be contiguous and hold the span the call touches, or the call
raises before any pointer reaches the library.  No GPU needed."""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc
from oracle import alltoall as o_a2a


class _Dev:
    """Stands in for a contiguous CUDA tensor of `n` elements of `esize` bytes.
    Its address is never dereferenced: a call it reaches either fails a span
    check in the binding or reaches the library without a communicator, which
    every collective entry point rejects before reading a pointer."""
    is_cuda = True

    def __init__(self, n, esize=4, shape=None):
        self.n, self.es = int(n), esize
        self.shape = shape or (self.n,)

    def numel(self):
        return self.n

    def element_size(self):
        return self.es

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 0x1000


def _comm(k):
    c = object.__new__(hoc.Comm)  # never initialised: the library answers ERR_NOT_INITIALIZED
    c.k, c._h = k, None
    return c


def _reaches_library(call):
    with pytest.raises(hoc.HocError) as e:
        call()
    assert e.value.code == hoc.ERR_NOT_INITIALIZED


def test_short_rank_buffer_is_named():
    c = _comm(4)
    recv = [_Dev(100) for _ in range(4)]
    recv[2] = _Dev(99)
    with pytest.raises(ValueError, match=r"recv\[2\]: tensor holds 396 bytes, the call touches 400"):
        c.allreduce([_Dev(100)] * 4, recv, dtype=hoc.FLOAT32)
    _reaches_library(lambda: c.allreduce([_Dev(100)] * 4, [_Dev(100)] * 4, dtype=hoc.FLOAT32, stream=0))
    # a count smaller than the tensors is fine; a larger one is not
    _reaches_library(lambda: c.allreduce([_Dev(100)] * 4, [_Dev(100)] * 4, count=60, dtype=hoc.FLOAT32, stream=0))
    with pytest.raises(ValueError, match=r"send\[0\]"):
        c.allreduce([_Dev(100)] * 4, [_Dev(100)] * 4, count=101, dtype=hoc.FLOAT32)


def test_non_contiguous_cpu_and_wrong_rank_count():
    c = _comm(2)
    strided = torch.zeros(10, 20)[:, 0]
    with pytest.raises(ValueError, match="contiguous"):
        c.allreduce([strided, _Dev(10)], [_Dev(10)] * 2, dtype=hoc.FLOAT32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        c.allreduce([torch.zeros(10)] * 2, [_Dev(10)] * 2, dtype=hoc.FLOAT32)
    with pytest.raises(ValueError, match="expected 2 rank buffers, got 3"):
        c.allreduce([_Dev(10)] * 3, [_Dev(10)] * 3, dtype=hoc.FLOAT32)


def test_reduce_scatter_and_allgather_spans_are_k_blocks():
    k, n = 4, 8
    c = _comm(k)
    with pytest.raises(ValueError, match=r"send\[0\]: tensor holds 124 bytes, the call touches 128"):
        c.reduce_scatter([_Dev(k * n - 1)] + [_Dev(k * n)] * (k - 1), [_Dev(n)] * k, dtype=hoc.FLOAT32)
    _reaches_library(lambda: c.reduce_scatter([_Dev(k * n)] * k, [_Dev(n)] * k, dtype=hoc.FLOAT32, stream=0))
    with pytest.raises(ValueError, match=r"recv\[3\]: .* the call touches 64"):
        c.allgather([_Dev(n, 2)] * k, [_Dev(k * n, 2)] * (k - 1) + [_Dev(k * n - 1, 2)], dtype=hoc.BFLOAT16)
    _reaches_library(lambda: c.allgather([_Dev(n, 2)] * k, [_Dev(k * n, 2)] * k, dtype=hoc.BFLOAT16, stream=0))


@pytest.mark.parametrize("custom_rdispls", [False, True])
def test_alltoall_spans_follow_the_displacements(custom_rdispls):
    k = 4
    rng = np.random.default_rng(7)
    counts = rng.integers(0, 9, size=(k, k))
    counts[1, 2] = 0                                   # an empty flow
    sd, rd = o_a2a.default_displs(counts)
    if custom_rdispls:                                 # segments in reverse source order, gaps of 3
        rd = np.zeros((k, k), dtype=np.int64)
        for d in range(k):
            at = 3
            for s in reversed(range(k)):
                rd[d][s] = at
                at += counts[s][d] + 3
    # spans from the oracle's layout: the end of each rank's furthest segment
    send_len = [int(max(sd[s][d] + counts[s][d] for d in range(k))) for s in range(k)]
    recv_len = [int(max(rd[d][s] + counts[s][d] for s in range(k))) for d in range(k)]
    c = _comm(k)
    kw = dict(sendcounts=counts, rdispls=rd if custom_rdispls else None, dtype=hoc.FLOAT32)
    _reaches_library(lambda: c.alltoall([_Dev(n) for n in send_len], [_Dev(n) for n in recv_len], **kw, stream=0))
    for d in range(k):
        short = [_Dev(n - (1 if i == d else 0)) for i, n in enumerate(recv_len)]
        with pytest.raises(ValueError, match=rf"recv\[{d}\]: tensor holds"):
            c.alltoall([_Dev(n) for n in send_len], short, **kw)
    for s in range(k):
        short = [_Dev(n - (1 if i == s else 0)) for i, n in enumerate(send_len)]
        with pytest.raises(ValueError, match=rf"send\[{s}\]: tensor holds"):
            c.alltoall(short, [_Dev(n) for n in recv_len], **kw)


def test_uniform_alltoall_span_is_k_counts():
    c = _comm(3)
    with pytest.raises(ValueError, match=r"recv\[0\]: .* the call touches 60"):
        c.alltoall([_Dev(15)] * 3, [_Dev(14)] + [_Dev(15)] * 2, count=5, dtype=hoc.FLOAT32)
    _reaches_library(lambda: c.alltoall([_Dev(15)] * 3, [_Dev(15)] * 3, count=5, dtype=hoc.FLOAT32, stream=0))


def test_host_allreduce_takes_cpu_tensors_and_checks_spans():
    c = _comm(2)
    z = lambda n: torch.zeros(n, dtype=torch.float32)
    with pytest.raises(ValueError, match=r"h_recv\[1\]"):
        c.allreduce_host([z(16)] * 2, [z(16), z(15)])
    with pytest.raises(ValueError, match="CPU tensors"):
        c.allreduce_host([_Dev(16)] * 2, [z(16)] * 2, dtype=hoc.FLOAT32)
    _reaches_library(lambda: c.allreduce_host([z(16)] * 2, [z(16)] * 2, stream=0))


def test_module_level_calls_check_spans():
    with pytest.raises(ValueError, match=r"dst\[1\]: tensor holds 63 bytes, the call touches 64"):
        hoc.tma_moves_noalloc([_Dev(64, 1)] * 2, [_Dev(64, 1), _Dev(63, 1)], [64, 64])
    tokens, topk, hidden = 5, 2, 8
    n = tokens * topk
    with pytest.raises(ValueError, match="pos_of: tensor holds 36 bytes, the call touches 40"):
        hoc.ep_pack(_Dev(n), _Dev(tokens * hidden, 2, (tokens, hidden)), 4, 2, _Dev(n * hidden, 2), _Dev(n),
                    _Dev(n - 1), _Dev(2, 8), _Dev(64))
    with pytest.raises(ValueError, match="y: tensor holds"):
        hoc.ep_combine(_Dev(n * hidden, 2), _Dev(n), _Dev(n), tokens, topk, hidden, _Dev((tokens - 1) * hidden, 2))
    with pytest.raises(ValueError, match="src: tensor holds"):
        hoc.xor16(_Dev(9, 2), _Dev(10, 2), 10, 0x5A5A, stream=0)
