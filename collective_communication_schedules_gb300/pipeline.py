"""One-forward-one-backward pipeline over simulated stages on one GPU.

HOCCL section 2.1: pipeline parallelism overlaps the activation and gradient
transfers of one micro-batch with the forward or backward compute of another,
which is why its communication runs beside compute kernels.  Each stage here
has its own CUDA stream; a stage's compute is the FMA probe (its SM budget)
plus an exact XOR transform of the payload, and every activation / gradient
hand-off is one send/recv from the producing stage's buffer into the
consuming stage's buffer (section 3.3.2, direct copy into the receiver).
Cross-stage order uses CUDA events only.  Three ways to hand over a buffer:
sends="stream": hoc_sendrecv on the producing stage's stream, which then
waits for the copy before its next compute; sends="event":
hoc_sendrecv_async, the copy runs on a copy stream and completes an event the
consumer waits on (the producer is not held, but the hand-off crosses two
stream dependencies); sends="pull" (the default): the consuming stage waits
for the producer's compute and issues the copy on its own stream, so the
producer is not held and the hand-off crosses one dependency.

The schedule: stage s of p runs min(p - s - 1, m) warm-up forwards, then
alternates forward and backward, then drains its backwards.
"""
from __future__ import annotations

import torch

from . import hoc


def stage_order(p: int, m: int) -> list[list[tuple[str, int]]]:
    out = []
    for s in range(p):
        warm = min(p - s - 1, m)
        seq = [("F", i) for i in range(warm)]
        nf, nb = warm, 0
        while nb < m:
            if nf < m:
                seq.append(("F", nf))
                nf += 1
            seq.append(("B", nb))
            nb += 1
        out.append(seq)
    return out


class Pipeline1F1B:
    """Buffers and streams for p stages x m micro-batches of `elems` bf16 values."""

    def __init__(self, comm: hoc.Comm, p: int, m: int, elems: int, keys, probe_ctas: int = 0,
                 probe_iters: int = 0, device: int = 0, sentinel: int = 0xA5A5, sends: str = "pull"):
        if comm.k < p:
            raise ValueError("the communicator needs one simulated rank per stage")
        if sends not in ("pull", "event", "stream"):
            raise ValueError("sends is 'pull', 'event' or 'stream'")
        self.sends = sends
        self.comm, self.p, self.m, self.elems = comm, p, m, elems
        self.keys = [[(int(keys[s][i][0]), int(keys[s][i][1])) for i in range(m)] for s in range(p)]
        self.probe_ctas, self.probe_iters = probe_ctas, probe_iters
        dev = torch.device("cuda", device)

        def buf():
            return torch.full((elems,), sentinel - 65536 if sentinel > 32767 else sentinel,
                              dtype=torch.int16, device=dev)

        self.act_in = [[buf() for _ in range(m)] for _ in range(p)]
        self.act_out = [[buf() for _ in range(m)] for _ in range(p)]
        self.grad_in = [[buf() for _ in range(m)] for _ in range(p)]
        self.grad_out = [[buf() for _ in range(m)] for _ in range(p)]
        self.streams = [torch.cuda.Stream(device=dev) for _ in range(p)]
        self.sent_f = [[None] * m for _ in range(p)]
        self.sent_b = [[None] * m for _ in range(p)]
        self.issue_trace = []

    def load(self, xs):
        for i, x in enumerate(xs):
            self.act_in[0][i].copy_(x.view(torch.int16) if x.dtype != torch.int16 else x)

    def _compute(self, s, src, dst, key, weight):
        st = self.streams[s]
        if self.probe_ctas and self.probe_iters:
            hoc.probe_launch(self.probe_ctas, 256, weight * self.probe_iters, stream=st)
        hoc.xor16(src, dst, self.elems, key, stream=st)

    def _forward(self, s, i):
        st = self.streams[s]
        if s > 0:
            st.wait_event(self.sent_f[s - 1][i])
            if self.sends == "pull":
                self.comm.sendrecv(s - 1, self.act_out[s - 1][i], s, self.act_in[s][i], self.elems, hoc.BFLOAT16,
                                   stream=st)
        self._compute(s, self.act_in[s][i], self.act_out[s][i], self.keys[s][i][0], 1)
        self.sent_f[s][i] = self._send(st, s, self.act_out[s][i], s + 1, self.act_in[s + 1][i] if s + 1 < self.p else None)

    def _backward(self, s, i):
        st = self.streams[s]
        if s + 1 < self.p:
            st.wait_event(self.sent_b[s + 1][i])
            if self.sends == "pull":
                self.comm.sendrecv(s + 1, self.grad_out[s + 1][i], s, self.grad_in[s][i], self.elems, hoc.BFLOAT16,
                                   stream=st)
            src = self.grad_in[s][i]
        else:
            src = self.act_out[s][i]         # the last stage starts from its own forward output
        self._compute(s, src, self.grad_out[s][i], self.keys[s][i][1], 2)
        self.sent_b[s][i] = self._send(st, s, self.grad_out[s][i], s - 1, self.grad_in[s - 1][i] if s > 0 else None)

    def _send(self, st, s, src, d, dst):
        """Hand `src` to stage d's `dst` after stage s's work so far; returns the event its consumer waits on
        (the stage's own progress when there is nothing to send)."""
        ev = torch.cuda.Event()
        if dst is None or self.sends == "pull":       # pull: the consumer issues the copy after this event
            ev.record(st)
        elif self.sends == "event":
            self.comm.sendrecv_async(s, src, d, dst, self.elems, hoc.BFLOAT16, stream=st, done=ev)
        else:
            self.comm.sendrecv(s, src, d, dst, self.elems, hoc.BFLOAT16, stream=st)
            ev.record(st)
        return ev

    def issue(self, origin: torch.cuda.Stream | None = None):
        """Issue every stage's operations; an operation is issued once the
        operation it depends on has been issued (its event then exists)."""
        origin = origin or torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(origin)
        for st in self.streams:
            st.wait_event(start)
        order = stage_order(self.p, self.m)
        pc = [0] * self.p
        issued_f = [[False] * self.m for _ in range(self.p)]
        issued_b = [[False] * self.m for _ in range(self.p)]
        remaining = sum(len(o) for o in order)
        while remaining:
            progress = False
            for s in range(self.p):
                if pc[s] >= len(order[s]):
                    continue
                kind, i = order[s][pc[s]]
                if kind == "F":
                    if s > 0 and not issued_f[s - 1][i]:
                        continue
                    self._forward(s, i)
                    issued_f[s][i] = True
                else:
                    if s + 1 < self.p and not issued_b[s + 1][i]:
                        continue
                    if s + 1 == self.p and not issued_f[s][i]:
                        continue
                    self._backward(s, i)
                    issued_b[s][i] = True
                self.issue_trace.append((s, kind, i))
                pc[s] += 1
                remaining -= 1
                progress = True
            if not progress:
                raise RuntimeError("1F1B issue order deadlocked")
        for st in self.streams:
            ev = torch.cuda.Event()
            ev.record(st)
            origin.wait_event(ev)

    def result(self, i: int) -> torch.Tensor:
        return self.grad_out[0][i]
