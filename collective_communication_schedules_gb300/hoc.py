"""Python binding of libhoc.so (ctypes).  Argument marshalling only.

Every collective runs in the library's CUDA kernels and copy-engine copies;
this module converts tensors (or raw device pointers) and streams into the
C ABI declared in include/hoc.h and turns result codes into exceptions.  If
the library is missing it raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhoc.so")

SUCCESS, ERR_INVALID_ARG, ERR_CUDA, ERR_OOM, ERR_NOT_INITIALIZED, ERR_UNSUPPORTED, ERR_TIMEOUT, ERR_NO_DEVICE = range(8)
INT32, FLOAT32, BFLOAT16, UINT8 = 0, 1, 2, 3
SUM = 0
PATH_AUTO, PATH_CE, PATH_TMA, PATH_FUSED = 0, 1, 2, 3
KERNEL_REDUCE, KERNEL_FUSED, KERNEL_TMA = 0, 1, 2
OP_ALLREDUCE, OP_REDUCE_SCATTER, OP_ALLGATHER, OP_ALLTOALL, OP_SENDRECV = range(5)
ITEM_REDUCE, ITEM_FUSED, ITEM_COPY, ITEM_TMA, ITEM_JOIN = range(5)
BUF_SEND, BUF_RECV = 0, 1
MAX_RANKS = 16
PATHS = {"auto": PATH_AUTO, "ce": PATH_CE, "tma": PATH_TMA, "fused": PATH_FUSED}
REDUCE_AUTO, REDUCE_LSU, REDUCE_TMA = 0, 1, 2
ENGINES = {"auto": REDUCE_AUTO, "lsu": REDUCE_LSU, "tma": REDUCE_TMA}


class HocError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} ({code}): {detail}")


class _Config(C.Structure):
    _fields_ = [("path", C.c_int), ("chunk_bytes", C.c_size_t), ("n_copy_streams", C.c_int),
                ("pipeline_depth", C.c_int), ("reduce_max_sms", C.c_int), ("copy_max_sms", C.c_int),
                ("use_graphs", C.c_int), ("a2a_interleave", C.c_int), ("a2a_stage_sync", C.c_int),
                ("ring_order", C.POINTER(C.c_int)), ("reduce_engine", C.c_int)]


class _Stats(C.Structure):
    _fields_ = [("path", C.c_int), ("kernels", C.c_int), ("copies", C.c_int), ("max_ctas", C.c_int),
                ("sms_used", C.c_int), ("graph_replayed", C.c_int), ("bytes_exec", C.c_size_t),
                ("bytes_min", C.c_size_t)]


class _PlanItem(C.Structure):
    _fields_ = [("kind", C.c_int), ("step", C.c_int), ("stream", C.c_int), ("stage", C.c_int),
                ("src_rank", C.c_int), ("dst_rank", C.c_int), ("src_buf", C.c_int), ("dst_buf", C.c_int),
                ("src_off", C.c_size_t), ("dst_off", C.c_size_t), ("bytes", C.c_size_t),
                ("n_waits", C.c_int), ("wait0", C.c_int)]


class _StepTime(C.Structure):
    _fields_ = [("kind", C.c_int), ("stream", C.c_int), ("stage", C.c_int), ("start_ms", C.c_float),
                ("end_ms", C.c_float)]


_lib = None

# Exported symbol -> (restype, argtypes)
_SIGS = {
    "hoc_config_default": (C.c_int, [C.POINTER(_Config)]),
    "hoc_init": (C.c_int, [C.POINTER(C.c_void_p), C.c_int, C.c_int, C.POINTER(_Config)]),
    "hoc_destroy": (C.c_int, [C.c_void_p]),
    "hoc_allreduce": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_size_t, C.c_int,
                                C.c_int, C.c_void_p]),
    "hoc_reduce_scatter": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_size_t,
                                     C.c_int, C.c_int, C.c_void_p]),
    "hoc_allgather": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_size_t, C.c_int,
                                C.c_void_p]),
    "hoc_alltoall": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_size_t), C.POINTER(C.c_size_t),
                               C.POINTER(C.c_void_p), C.POINTER(C.c_size_t), C.c_size_t, C.c_int, C.c_void_p]),
    "hoc_sendrecv": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_size_t, C.c_int,
                               C.c_void_p]),
    "hoc_sendrecv_async": (C.c_int, [C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p, C.c_size_t, C.c_int,
                                     C.c_void_p, C.c_void_p]),
    "hoc_wait": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int]),
    "hoc_last_stats": (C.c_int, [C.c_void_p, C.POINTER(_Stats)]),
    "hoc_profile_enable": (C.c_int, [C.c_void_p, C.c_int]),
    "hoc_profile_read": (C.c_int, [C.c_void_p, C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_double)]),
    "hoc_error_string": (C.c_char_p, [C.c_int]),
    "hoc_last_error_detail": (C.c_char_p, []),
    "hoc_plan_query": (C.c_int, [C.c_int, C.POINTER(_Config), C.c_int, C.c_size_t, C.c_int, C.POINTER(C.c_size_t),
                                 C.POINTER(_PlanItem), C.c_size_t, C.POINTER(C.c_size_t)]),
    "hoc_probe_launch": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p]),
    "hoc_xor16_launch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_uint16]),
    "hoc_device_sm_count": (C.c_int, [C.c_int, C.POINTER(C.c_int)]),
    "hoc_tma_moves_noalloc": (C.c_int, [C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.POINTER(C.c_size_t),
                                        C.c_int, C.c_int, C.c_void_p, C.c_int]),
}
NOALLOC_MAX_MOVES = 192
_SIGS["hoc_alltoall_device_counts"] = (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                                 C.c_void_p, C.c_int, C.POINTER(C.c_size_t), C.POINTER(C.c_size_t),
                                                 C.c_int, C.c_void_p])
_SIGS["hoc_ep_pack"] = (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                  C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p])
_SIGS["hoc_ep_pack_workspace"] = (C.c_int, [C.c_int, C.c_int, C.c_int, C.POINTER(C.c_size_t)])
_SIGS["hoc_ep_combine"] = (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p,
                                     C.c_void_p])
_SIGS["hoc_ep_dispatch_fused"] = (C.c_int, [C.c_int, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int, C.c_int,
                                            C.c_int, C.c_int, C.POINTER(C.c_void_p), C.POINTER(C.c_size_t),
                                            C.POINTER(C.c_void_p), C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p,
                                            C.c_void_p])
_SIGS["hoc_ep_combine_fused"] = (C.c_int, [C.c_int, C.POINTER(C.c_void_p), C.POINTER(C.c_size_t),
                                           C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_void_p,
                                           C.POINTER(C.c_void_p), C.c_int, C.c_int, C.c_int, C.c_int,
                                           C.POINTER(C.c_void_p), C.c_void_p, C.c_void_p])
_SIGS["hoc_ep_pack_all"] = _SIGS["hoc_ep_dispatch_fused"]
_SIGS["hoc_ep_combine_all"] = (C.c_int, [C.c_int, C.POINTER(C.c_void_p), C.POINTER(C.c_size_t), C.POINTER(C.c_void_p),
                                         C.POINTER(C.c_void_p), C.c_int, C.c_int, C.c_int, C.POINTER(C.c_void_p),
                                         C.c_void_p, C.c_void_p])
_SIGS["hoc_allreduce_host"] = (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_size_t,
                                         C.c_int, C.c_int, C.c_void_p])
_SIGS["hoc_proxy_status"] = (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64),
                                       C.POINTER(C.c_int)])
_SIGS["hoc_profile_stream_finish"] = (C.c_int, [C.c_void_p, C.POINTER(C.c_float), C.c_int, C.POINTER(C.c_int)])
_SIGS["hoc_profile_timeline"] = (C.c_int, [C.c_void_p, C.POINTER(_StepTime), C.c_size_t, C.POINTER(C.c_size_t)])
_SIGS["hoc_topo_schedule"] = (C.c_int, [C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int), C.POINTER(C.c_uint64),
                                        C.c_uint64, C.c_uint64, C.POINTER(C.c_uint64), C.POINTER(C.c_uint64),
                                        C.POINTER(C.c_double), C.c_int, C.POINTER(C.c_int),
                                        C.POINTER(C.c_double)])


def lib():
    """Load libhoc.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m collective_communication_schedules_gb300.build`")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def error_string(code: int) -> str:
    return lib().hoc_error_string(code).decode()


def last_error_detail() -> str:
    return lib().hoc_last_error_detail().decode()


def _check(code: int, where: str):
    if code != SUCCESS:
        raise HocError(code, where, last_error_detail())


# ----------------------------------------------------------------- marshalling
def _dtype_code(x) -> int:
    import torch
    m = {torch.int32: INT32, torch.float32: FLOAT32, torch.bfloat16: BFLOAT16, torch.uint8: UINT8}
    if x.dtype not in m:
        raise TypeError(f"unsupported tensor dtype {x.dtype}")
    return m[x.dtype]


DTYPE_BYTES = {INT32: 4, FLOAT32: 4, BFLOAT16: 2, UINT8: 1}


def _ptr(x, nbytes: int = 0, what: str = "buffer", device: bool = True) -> int:
    """Address of `x`.  A tensor must be contiguous, hold at least `nbytes`
    bytes (the span the call touches) and live on the GPU (`device`) or the
    host; an int is taken as a raw address, unchecked."""
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError(f"{what}: tensor must be contiguous")
    have = x.numel() * x.element_size()
    if have < nbytes:
        raise ValueError(f"{what}: tensor holds {have} bytes, the call touches {nbytes}")
    if device and not x.is_cuda:
        raise ValueError(f"{what}: rank buffers must be CUDA tensors")
    if not device and x.is_cuda:
        raise ValueError(f"{what}: host buffers must be CPU tensors")
    return x.data_ptr()


def _ptr_array(xs: Sequence, nbytes=0, what: str = "buffer", device: bool = True) -> C.Array:
    """Addresses of the rank buffers; `nbytes` is one span for all ranks or a list, one per rank."""
    spans = list(nbytes) if isinstance(nbytes, (list, tuple)) else [nbytes] * len(xs)
    if len(spans) != len(xs):
        raise ValueError(f"{what}: expected {len(spans)} rank buffers, got {len(xs)}")
    return (C.c_void_p * len(xs))(*[_ptr(x, n, f"{what}[{r}]", device) for r, (x, n) in enumerate(zip(xs, spans))])


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _sizes(vals, n) -> Optional[C.Array]:
    if vals is None:
        return None
    flat = [int(v) for row in vals for v in (row if hasattr(row, "__len__") else [row])]
    if len(flat) != n:
        raise ValueError(f"expected {n} values, got {len(flat)}")
    return (C.c_size_t * n)(*flat)


@dataclass
class Config:
    path: str = "auto"
    chunk_bytes: int = 0  # 0: picked by the scheduler (allreduce: by move path and rank count)
    n_copy_streams: int = 0  # 0: the scheduler picks per call (8 queues for copies of at most 2 MiB, else 4)
    pipeline_depth: int = 0
    reduce_max_sms: int = 0
    copy_max_sms: int = 0
    use_graphs: bool = True
    a2a_interleave: bool = True
    a2a_stage_sync: bool = False
    ring_order: Optional[Sequence[int]] = None
    reduce_engine: str = "auto"
    _keep: list = field(default_factory=list, repr=False)

    def to_c(self) -> _Config:
        c = _Config()
        c.path = PATHS[self.path] if isinstance(self.path, str) else int(self.path)
        c.chunk_bytes = int(self.chunk_bytes)
        c.n_copy_streams = int(self.n_copy_streams)
        c.pipeline_depth = int(self.pipeline_depth)
        c.reduce_max_sms = int(self.reduce_max_sms)
        c.copy_max_sms = int(self.copy_max_sms)
        c.use_graphs = int(bool(self.use_graphs))
        c.a2a_interleave = int(bool(self.a2a_interleave))
        c.a2a_stage_sync = int(bool(self.a2a_stage_sync))
        c.reduce_engine = ENGINES[self.reduce_engine] if isinstance(self.reduce_engine, str) else int(self.reduce_engine)
        if self.ring_order is not None:
            arr = (C.c_int * len(self.ring_order))(*[int(v) for v in self.ring_order])
            self._keep = [arr]
            c.ring_order = C.cast(arr, C.POINTER(C.c_int))
        else:
            c.ring_order = None
        return c


class Comm:
    """A communicator over `nranks` simulated ranks on one CUDA device."""

    def __init__(self, nranks: int, device: int = 0, config: Optional[Config] = None):
        self.k = nranks
        self.device = device
        self.config = config or Config()
        h = C.c_void_p()
        cfg = self.config.to_c()
        _check(lib().hoc_init(C.byref(h), nranks, device, C.byref(cfg)), "hoc_init")
        self._h = h

    def _ranks(self, xs, nbytes, what, device=True):
        if len(xs) != self.k:
            raise ValueError(f"{what}: expected {self.k} rank buffers, got {len(xs)}")
        return _ptr_array(xs, nbytes, what, device)

    def close(self):
        if getattr(self, "_h", None):
            _check(lib().hoc_destroy(self._h), "hoc_destroy")
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ collectives
    def allreduce(self, send, recv, count=None, dtype=None, stream=None):
        count = send[0].numel() if count is None else count
        dtype = _dtype_code(send[0]) if dtype is None else dtype
        n = int(count) * DTYPE_BYTES[dtype]
        _check(lib().hoc_allreduce(self._h, self._ranks(send, n, "send"), self._ranks(recv, n, "recv"), count, dtype,
                                   SUM, _stream(stream)), "hoc_allreduce")

    def allreduce_host(self, h_send, h_recv, count=None, dtype=None, stream=None):
        """AllReduce of host (CPU) tensors: one fused launch on host memory the GPU can address (path AUTO/FUSED),
        else the copy-engine pipeline through device staging slots (path CE/TMA)."""
        count = h_send[0].numel() if count is None else count
        dtype = _dtype_code(h_send[0]) if dtype is None else dtype
        n = int(count) * DTYPE_BYTES[dtype]
        _check(lib().hoc_allreduce_host(self._h, self._ranks(h_send, n, "h_send", device=False),
                                        self._ranks(h_recv, n, "h_recv", device=False), count, dtype, SUM,
                                        _stream(stream)), "hoc_allreduce_host")

    def reduce_scatter(self, send, recv, recvcount=None, dtype=None, stream=None):
        recvcount = recv[0].numel() if recvcount is None else recvcount
        dtype = _dtype_code(send[0]) if dtype is None else dtype
        n = int(recvcount) * DTYPE_BYTES[dtype]
        _check(lib().hoc_reduce_scatter(self._h, self._ranks(send, self.k * n, "send"), self._ranks(recv, n, "recv"),
                                        recvcount, dtype, SUM, _stream(stream)), "hoc_reduce_scatter")

    def allgather(self, send, recv, sendcount=None, dtype=None, stream=None):
        sendcount = send[0].numel() if sendcount is None else sendcount
        dtype = _dtype_code(send[0]) if dtype is None else dtype
        n = int(sendcount) * DTYPE_BYTES[dtype]
        _check(lib().hoc_allgather(self._h, self._ranks(send, n, "send"), self._ranks(recv, self.k * n, "recv"),
                                   sendcount, dtype, _stream(stream)), "hoc_allgather")

    def alltoall(self, send, recv, sendcounts=None, sdispls=None, rdispls=None, count=0, dtype=None,
                 stream=None):
        """sendcounts: k x k (row = source) in elements; None = uniform `count`."""
        dtype = _dtype_code(send[0]) if dtype is None else dtype
        k, kk, b = self.k, self.k * self.k, DTYPE_BYTES[dtype]
        cnt = _sizes(sendcounts, kk)
        sd, rd = _sizes(sdispls, kk), _sizes(rdispls, kk)
        c = [cnt[i] for i in range(kk)] if cnt is not None else [int(count)] * kk
        # the span of each rank's buffer: the end of its furthest segment
        s_end = [max((sd[a * k + d] if sd is not None else sum(c[a * k: a * k + d])) + c[a * k + d]
                     for d in range(k)) * b for a in range(k)]
        r_end = [max((rd[d * k + a] if rd is not None else sum(c[x * k + d] for x in range(a))) + c[a * k + d]
                     for a in range(k)) * b for d in range(k)]
        _check(lib().hoc_alltoall(self._h, self._ranks(send, s_end, "send"), cnt, sd,
                                  self._ranks(recv, r_end, "recv"), rd, int(count), dtype, _stream(stream)),
               "hoc_alltoall")

    def sendrecv(self, src_rank, send, dst_rank, recv, count=None, dtype=None, stream=None):
        count = send.numel() if count is None else count
        dtype = _dtype_code(send) if dtype is None else dtype
        n = int(count) * DTYPE_BYTES[dtype]
        _check(lib().hoc_sendrecv(self._h, int(src_rank), _ptr(send, n, "send"), int(dst_rank), _ptr(recv, n, "recv"),
                                  count, dtype, _stream(stream)), "hoc_sendrecv")

    def sendrecv_async(self, src_rank, send, dst_rank, recv, count=None, dtype=None, stream=None, done=None):
        """Send/recv completed by an event, not by `stream`: returns the torch.cuda.Event (`done`, or a new
        one) that the consumer waits on; later work on `stream` does not wait for the copy."""
        import torch
        count = send.numel() if count is None else count
        dtype = _dtype_code(send) if dtype is None else dtype
        if done is None:
            done = torch.cuda.Event()
        if not done.cuda_event:
            done.record(torch.cuda.current_stream() if stream is None else stream)   # creates the CUDA event
        n = int(count) * DTYPE_BYTES[dtype]
        _check(lib().hoc_sendrecv_async(self._h, int(src_rank), _ptr(send, n, "send"), int(dst_rank),
                                        _ptr(recv, n, "recv"), count, dtype, _stream(stream),
                                        C.c_void_p(done.cuda_event)), "hoc_sendrecv_async")
        return done

    def alltoall_device_counts(self, send, recv, d_counts, recv_capacity, dtype=None, stream=None,
                               transpose: bool = False, send_capacity=None):
        """All-to-all(v) whose k x k counts (uint64/int64, elements, row = source) live on the device.

        The counts reach a host proxy through the stream-memory-operation
        handshake; the call returns without waiting (see include/hoc_proxy.h).
        send_capacity defaults to the elements each send tensor holds."""
        dtype = _dtype_code(send[0]) if dtype is None else dtype
        caps = [int(v) for v in recv_capacity]
        if len(caps) != self.k:
            raise ValueError(f"recv_capacity: expected {self.k} values, got {len(caps)}")
        if send_capacity is None:
            scaps = [t.numel() * t.element_size() // DTYPE_BYTES[dtype] if not isinstance(t, int) else None
                     for t in send]
            if any(v is None for v in scaps):
                raise ValueError("send_capacity is needed when send buffers are raw addresses")
        else:
            scaps = [int(v) for v in send_capacity]
        if len(scaps) != self.k:
            raise ValueError(f"send_capacity: expected {self.k} values, got {len(scaps)}")
        cap = (C.c_size_t * self.k)(*caps)
        scap = (C.c_size_t * self.k)(*scaps)
        _check(lib().hoc_alltoall_device_counts(self._h,
                                                self._ranks(send, [v * DTYPE_BYTES[dtype] for v in scaps], "send"),
                                                self._ranks(recv, [v * DTYPE_BYTES[dtype] for v in caps], "recv"),
                                                _ptr(d_counts, 8 * self.k * self.k, "d_counts"),
                                                int(bool(transpose)), scap, cap, dtype, _stream(stream)),
               "hoc_alltoall_device_counts")

    def proxy_status(self) -> dict:
        done = C.c_uint64()
        rel = C.c_uint64()
        err = C.c_int()
        _check(lib().hoc_proxy_status(self._h, C.byref(done), C.byref(rel), C.byref(err)), "hoc_proxy_status")
        return {"completed": done.value, "released_on_error": rel.value, "first_error": err.value}

    # ------------------------------------------------------------- control
    def wait(self, stream=None, timeout_ms: int = 60000):
        _check(lib().hoc_wait(self._h, _stream(stream), int(timeout_ms)), "hoc_wait")

    def last_stats(self) -> dict:
        s = _Stats()
        _check(lib().hoc_last_stats(self._h, C.byref(s)), "hoc_last_stats")
        return {name: getattr(s, name) for name, _ in _Stats._fields_}

    def profile_enable(self, on: bool = True):
        _check(lib().hoc_profile_enable(self._h, int(bool(on))), "hoc_profile_enable")

    def profile_read(self, kernel: int):
        n = C.c_int()
        ms = C.c_double()
        _check(lib().hoc_profile_read(self._h, int(kernel), C.byref(n), C.byref(ms)), "hoc_profile_read")
        return n.value, ms.value

    def profile_stream_finish(self) -> list:
        """Finish time (ms from the fork) of each copy stream of the last call issued while profiling."""
        buf = (C.c_float * 16)()
        n = C.c_int()
        _check(lib().hoc_profile_stream_finish(self._h, buf, 16, C.byref(n)), "hoc_profile_stream_finish")
        return [buf[i] for i in range(min(n.value, 16))]

    def profile_timeline(self) -> list:
        """Per-step (kind, stream, stage, start_ms, end_ms) of the last call issued while profiling."""
        n = C.c_size_t()
        _check(lib().hoc_profile_timeline(self._h, None, 0, C.byref(n)), "hoc_profile_timeline")
        buf = (_StepTime * max(1, n.value))()
        _check(lib().hoc_profile_timeline(self._h, buf, n.value, C.byref(n)), "hoc_profile_timeline")
        kinds = {ITEM_REDUCE: "reduce", ITEM_FUSED: "fused", ITEM_COPY: "copy", ITEM_TMA: "tma"}
        return [dict(kind=kinds.get(b.kind, b.kind), stream=b.stream, stage=b.stage, start_ms=b.start_ms,
                     end_ms=b.end_ms) for b in buf[: n.value]]


# ---------------------------------------------------------------- workload
PROBE_WHOLE_SM, PROBE_PDL = 1, 2


def probe_launch(ctas: int, threads: int, iters: int, sink=None, stream=None, whole_sm: bool = False,
                 pdl: bool = False):
    flags = (PROBE_WHOLE_SM if whole_sm else 0) | (PROBE_PDL if pdl else 0)
    _check(lib().hoc_probe_launch(_stream(stream), int(ctas), int(threads), int(iters), flags,
                                  None if sink is None else _ptr(sink, 12, "sink")), "hoc_probe_launch")


def xor16(src, dst, n: int, key: int, stream=None):
    _check(lib().hoc_xor16_launch(_stream(stream), _ptr(src, 2 * int(n), "src"), _ptr(dst, 2 * int(n), "dst"), int(n),
                                  int(key) & 0xFFFF), "hoc_xor16_launch")


def tma_moves_noalloc(src, dst, nbytes, max_ctas: int = 0, stream=None, wait: bool = True):
    """Byte moves src[i] -> dst[i] on the TMA bulk-copy kernel with no device
    allocation (for callers that cannot call cudaMalloc); see include/hoc.h."""
    n = len(nbytes)
    if len(src) != n or len(dst) != n:
        raise ValueError("src, dst and nbytes must have the same length")
    spans = [int(b) for b in nbytes]
    sizes = (C.c_size_t * max(1, n))(*spans)
    _check(lib().hoc_tma_moves_noalloc(_ptr_array(src, spans, "src"), _ptr_array(dst, spans, "dst"), sizes, n,
                                       int(max_ctas), _stream(stream), int(bool(wait))), "hoc_tma_moves_noalloc")


def topo_schedule(C_matrix, node_of, sym, bw_nvlink: int, bw_rdma: int):
    """Two-domain stage schedule (host only): returns (T, stages, taus, total)."""
    G = len(node_of)
    flat = [int(v) for row in C_matrix for v in row]
    if len(flat) != G * G:
        raise ValueError("C must be G x G")
    cm = (C.c_uint64 * (G * G))(*flat)
    no = (C.c_int * G)(*[int(v) for v in node_of])
    sy = (C.c_int * G)(*[int(v) for v in sym])
    n = C.c_int()
    tot = C.c_double()
    _check(lib().hoc_topo_schedule(G, no, sy, cm, int(bw_nvlink), int(bw_rdma), None, None, None, 0, C.byref(n),
                                   C.byref(tot)), "hoc_topo_schedule")
    T = (C.c_uint64 * (G * G))()
    st = (C.c_uint64 * max(1, n.value * G * G))()
    ta = (C.c_double * max(1, n.value))()
    _check(lib().hoc_topo_schedule(G, no, sy, cm, int(bw_nvlink), int(bw_rdma), T, st, ta, n.value, C.byref(n),
                                   C.byref(tot)), "hoc_topo_schedule")
    Tm = [[T[u * G + v] for v in range(G)] for u in range(G)]
    stages = [[[st[s * G * G + u * G + v] for v in range(G)] for u in range(G)] for s in range(n.value)]
    return Tm, stages, [ta[s] for s in range(n.value)], tot.value


def ep_pack_workspace(tokens: int, topk: int, experts: int) -> int:
    """int32 entries of scratch that ep_pack needs for this shape."""
    n = C.c_size_t()
    _check(lib().hoc_ep_pack_workspace(int(tokens), int(topk), int(experts), C.byref(n)), "hoc_ep_pack_workspace")
    return n.value


def ep_pack(expert_ids, x, experts: int, nranks: int, send, perm, pos_of, dst_counts, workspace, stream=None):
    """Dispatch-side pack of one source rank (device tensors; see include/hoc_ep.h)."""
    tokens, hidden = x.shape
    topk = expert_ids.numel() // tokens if tokens else 1
    n = tokens * topk
    _check(lib().hoc_ep_pack(_ptr(expert_ids, 4 * n, "expert_ids"), _ptr(x, 2 * tokens * hidden, "x"), int(tokens),
                             int(topk), int(hidden), int(experts), int(nranks), _ptr(send, 2 * n * hidden, "send"),
                             _ptr(perm, 4 * n, "perm"), _ptr(pos_of, 4 * n, "pos_of"),
                             _ptr(dst_counts, 8 * int(nranks), "dst_counts"), _ptr(workspace, 0, "workspace"),
                             int(workspace.numel()), _stream(stream)), "hoc_ep_pack")


def ep_combine(rows, pos_of, weights, tokens: int, topk: int, hidden: int, y, stream=None):
    """Gate-weighted top-k combine of one source rank (see include/hoc_ep.h)."""
    n = int(tokens) * int(topk)
    _check(lib().hoc_ep_combine(_ptr(rows, 2 * n * int(hidden), "rows"), _ptr(pos_of, 4 * n, "pos_of"),
                                _ptr(weights, 4 * n, "weights"), int(tokens), int(topk), int(hidden),
                                _ptr(y, 2 * int(tokens) * int(hidden), "y"), _stream(stream)), "hoc_ep_combine")


def _ep_scatter_call(fn_name, expert_ids, x, experts, out, out_capacity, pos_of, counts, workspace, status, stream):
    k = len(x)
    tokens, hidden = x[0].shape
    topk = expert_ids[0].numel() // tokens if tokens else 1
    n = tokens * topk
    caps = [int(v) for v in out_capacity]
    if len(caps) != k or len(expert_ids) != k or len(out) != k or len(pos_of) != k:
        raise ValueError(f"expected {k} per-rank tensors and capacities")
    cap = (C.c_size_t * k)(*caps)
    _check(getattr(lib(), fn_name)(k, _ptr_array(expert_ids, 4 * n, "expert_ids"),
                                   _ptr_array(x, 2 * tokens * hidden, "x"), int(tokens), int(topk), int(hidden),
                                   int(experts), _ptr_array(out, [2 * c for c in caps], "out"), cap,
                                   _ptr_array(pos_of, 4 * n, "pos_of"), _ptr(counts, 8 * k * k, "counts"),
                                   _ptr(workspace, 0, "workspace"), int(workspace.numel()),
                                   _ptr(status, 4, "status"), _stream(stream)), fn_name)


def ep_pack_all(expert_ids, x, experts: int, send, send_capacity, pos_of, counts, workspace, status, stream=None):
    """hoc_ep_pack for every source rank in one pass (see include/hoc_ep.h): lists of k device tensors."""
    _ep_scatter_call("hoc_ep_pack_all", expert_ids, x, experts, send, send_capacity, pos_of, counts, workspace,
                     status, stream)


def ep_combine_all(rows, rows_capacity, pos_of, weights, tokens: int, topk: int, hidden: int, y, status,
                   stream=None):
    """hoc_ep_combine for every source rank in one pass (see include/hoc_ep.h)."""
    k = len(rows)
    n = int(tokens) * int(topk)
    caps = [int(v) for v in rows_capacity]
    if len(caps) != k or len(pos_of) != k or len(weights) != k or len(y) != k:
        raise ValueError(f"expected {k} per-rank tensors and capacities")
    cap = (C.c_size_t * k)(*caps)
    _check(lib().hoc_ep_combine_all(k, _ptr_array(rows, [2 * c for c in caps], "rows"), cap,
                                    _ptr_array(pos_of, 4 * n, "pos_of"), _ptr_array(weights, 4 * n, "weights"),
                                    int(tokens), int(topk), int(hidden),
                                    _ptr_array(y, 2 * int(tokens) * int(hidden), "y"), _ptr(status, 4, "status"),
                                    _stream(stream)), "hoc_ep_combine_all")


def ep_dispatch_fused(expert_ids, x, experts: int, recv, recv_capacity, pos_of, counts, workspace, status,
                      stream=None):
    """Dispatch of every source rank straight into the receive buffers (see include/hoc_ep.h).

    Lists of k device tensors: expert_ids [tokens*topk] int32, x [tokens, hidden] bf16, recv (room for
    recv_capacity[d] elements each), pos_of [tokens*topk] int32; counts: [k, k] int64; status: int32."""
    k = len(x)
    tokens, hidden = x[0].shape
    topk = expert_ids[0].numel() // tokens if tokens else 1
    n = tokens * topk
    caps = [int(v) for v in recv_capacity]
    if len(caps) != k or len(expert_ids) != k or len(recv) != k or len(pos_of) != k:
        raise ValueError(f"expected {k} per-rank tensors and capacities")
    cap = (C.c_size_t * k)(*caps)
    _check(lib().hoc_ep_dispatch_fused(k, _ptr_array(expert_ids, 4 * n, "expert_ids"),
                                       _ptr_array(x, 2 * tokens * hidden, "x"), int(tokens), int(topk), int(hidden),
                                       int(experts), _ptr_array(recv, [2 * c for c in caps], "recv"), cap,
                                       _ptr_array(pos_of, 4 * n, "pos_of"), _ptr(counts, 8 * k * k, "counts"),
                                       _ptr(workspace, 0, "workspace"), int(workspace.numel()),
                                       _ptr(status, 4, "status"), _stream(stream)), "hoc_ep_dispatch_fused")


def ep_combine_fused(rows, rows_capacity, expert_ids, pos_of, counts, weights, tokens: int, topk: int, hidden: int,
                     experts: int, y, status, stream=None):
    """Combine of every source rank reading the expert ranks' rows in place (see include/hoc_ep.h)."""
    k = len(rows)
    n = int(tokens) * int(topk)
    caps = [int(v) for v in rows_capacity]
    if len(caps) != k or len(expert_ids) != k or len(pos_of) != k or len(weights) != k or len(y) != k:
        raise ValueError(f"expected {k} per-rank tensors and capacities")
    cap = (C.c_size_t * k)(*caps)
    _check(lib().hoc_ep_combine_fused(k, _ptr_array(rows, [2 * c for c in caps], "rows"), cap,
                                      _ptr_array(expert_ids, 4 * n, "expert_ids"), _ptr_array(pos_of, 4 * n, "pos_of"),
                                      _ptr(counts, 8 * k * k, "counts"), _ptr_array(weights, 4 * n, "weights"),
                                      int(tokens), int(topk), int(hidden), int(experts),
                                      _ptr_array(y, 2 * int(tokens) * int(hidden), "y"), _ptr(status, 4, "status"),
                                      _stream(stream)), "hoc_ep_combine_fused")


def sm_count(device: int = 0) -> int:
    n = C.c_int()
    _check(lib().hoc_device_sm_count(int(device), C.byref(n)), "hoc_device_sm_count")
    return n.value


def plan_query(nranks: int, op: int, count: int, dtype: int, counts=None, config: Optional[Config] = None):
    """The plan the scheduler would run, as a list of dicts (host only, no GPU)."""
    cfg = (config or Config()).to_c()
    cnt = _sizes(counts, nranks * nranks) if counts is not None else None
    n = C.c_size_t()
    _check(lib().hoc_plan_query(nranks, C.byref(cfg), op, int(count), dtype, cnt, None, 0, C.byref(n)),
           "hoc_plan_query")
    items = (_PlanItem * max(1, n.value))()
    _check(lib().hoc_plan_query(nranks, C.byref(cfg), op, int(count), dtype, cnt, items, n.value, C.byref(n)),
           "hoc_plan_query")
    return [{name: getattr(items[i], name) for name, _ in _PlanItem._fields_} for i in range(n.value)]
