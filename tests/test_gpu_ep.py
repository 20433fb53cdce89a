"""EP pack / combine kernels and the full dispatch-combine round trip on the GPU.

8 ranks x 4096 tokens x 2048 bf16, top-6 of 64 experts drawn from Zipf(1.1):
pack on the device, dispatch all-to-all with device-computed counts (host
proxy handshake), identity experts, combine all-to-all with the transposed
counts, weighted top-k combine -- all stream-ordered with no host sync, and
compared bit for bit with the oracle pipeline.
"""
import numpy as np
import pytest
import torch

from collective_communication_schedules_gb300 import hoc, inputs
from oracle import alltoall as o_a2a
from oracle import ep as o_ep
from tests.gpu_util import to_device, to_host

pytestmark = pytest.mark.gpu


def _rank_data(k, tokens, hidden, experts, topk, s):
    routing = inputs.ep_routing(k, tokens, experts, topk, s)
    xs = [inputs.normal_bf16(tokens * hidden, 5500 + r).reshape(tokens, hidden) for r in range(k)]
    rng = np.random.default_rng(5600)
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    return routing, xs, ws


def _pack_on_device(ids, x, experts, k, stream):
    tokens, hidden = x.shape
    n = ids.numel()
    send = torch.empty((n, hidden), dtype=torch.bfloat16, device="cuda")
    perm = torch.empty(n, dtype=torch.int32, device="cuda")
    pos_of = torch.empty(n, dtype=torch.int32, device="cuda")
    counts = torch.empty(k, dtype=torch.int64, device="cuda")
    ws = torch.empty(hoc.ep_pack_workspace(tokens, n // tokens, experts), dtype=torch.int32, device="cuda")
    hoc.ep_pack(ids, x, experts, k, send, perm, pos_of, counts, ws, stream=stream)
    return send, perm, pos_of, counts


@pytest.mark.parametrize("tokens,hidden,drop,experts,topk", [
    (4096, 2048, False, 64, 6),   # the EP workload's shape: 12 full tiles of 2048 pairs
    (333, 40, True, 64, 6),       # one partial tile, dropped pairs
    (5000, 64, True, 96, 4),      # ragged last tile, experts not a power of two
    (700, 16, False, 2048, 2),    # more than 1024 experts: the one-CTA-per-expert sort
    (3000, 16, True, 1024, 8),    # 12 tiles x 1024 experts: histograms past the shared budget, scanned in place
    (5120, 16, True, 512, 8),     # 20 tiles x 512 experts: the separate scan, on its shared-memory copy
    (2048, 16, True, 1024, 8),    # 8 tiles x 1024 experts: the largest histograms the placement scans itself
    (200, 24, False, 64, 10),     # topk above the combine's batched loads
    (250, 36, True, 64, 6),       # hidden not a multiple of 8: scalar combine
    (100, 16, True, 64, 40),      # topk above a warp: the scatter takes its destinations 32 at a time
])
def test_pack_and_combine_match_oracle(tokens, hidden, drop, experts, topk):
    k = 8
    routing, xs, ws = _rank_data(k, tokens, hidden, experts, topk, 1.1)
    ids = routing[0].astype(np.int32)
    if drop:
        ids[3, 2] = -5
        ids[7, 0] = experts
    want_send, want_perm, want_pos, want_counts = o_ep.pack(xs[0], ids, experts, k)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d_ids = torch.from_numpy(ids).cuda()
        d_x = to_device(xs[0], "bfloat16")
        send, perm, pos_of, counts = _pack_on_device(d_ids, d_x, experts, k, s)
    s.synchronize()
    nv = len(want_perm)
    assert np.array_equal(perm.cpu().numpy()[:nv], want_perm)
    assert np.all(perm.cpu().numpy()[nv:] == -1)
    assert np.array_equal(pos_of.cpu().numpy(), want_pos)
    assert np.array_equal(counts.cpu().numpy(), want_counts)
    assert np.array_equal(to_host(send, "bfloat16")[:nv], want_send)
    # combine of the packed rows themselves (identity experts, no exchange)
    y = torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda")
    w = torch.from_numpy(ws[0]).cuda()
    hoc.ep_combine(send, pos_of, w, tokens, topk, hidden, y)
    torch.cuda.synchronize()
    want_y = o_ep.combine(want_send, want_pos, ws[0], topk)
    assert np.array_equal(to_host(y, "bfloat16"), want_y)


def test_zero_tokens_is_a_no_op():
    k, hidden, experts = 8, 64, 64
    x = torch.empty((0, hidden), dtype=torch.bfloat16, device="cuda")
    ids = torch.empty(0, dtype=torch.int32, device="cuda")
    counts = torch.full((k,), 7, dtype=torch.int64, device="cuda")
    ws = torch.empty(max(1, hoc.ep_pack_workspace(0, 6, experts)), dtype=torch.int32, device="cuda")
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    hoc.ep_pack(ids, x, experts, k, torch.empty((0, hidden), dtype=torch.bfloat16, device="cuda"), empty, empty,
                counts, ws)
    y = torch.empty((0, hidden), dtype=torch.bfloat16, device="cuda")
    hoc.ep_combine(torch.empty((0, hidden), dtype=torch.bfloat16, device="cuda"), empty,
                   torch.empty(0, device="cuda"), 0, 6, hidden, y)
    torch.cuda.synchronize()
    assert counts.tolist() == [0] * k  # a rank without tokens sends nothing


def test_dispatch_combine_round_trip_without_host_sync():
    k, tokens, hidden, experts, topk = 8, 4096, 2048, 64, 6
    routing, xs, ws = _rank_data(k, tokens, hidden, experts, topk, 1.1)
    # oracle pipeline
    packs = [o_ep.pack(xs[r], routing[r], experts, k) for r in range(k)]
    counts = np.stack([p[3] for p in packs])
    sends = [p[0].reshape(-1) for p in packs]
    recv = o_a2a.alltoallv(sends, counts)
    back = o_a2a.alltoallv(recv, o_a2a.transpose_counts(counts))
    want_y = [o_ep.combine(back[r].reshape(-1, hidden), packs[r][2], ws[r], topk) for r in range(k)]
    # device pipeline on one stream
    s = torch.cuda.Stream()
    with hoc.Comm(k, 0) as c:
        with torch.cuda.stream(s):
            d_counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
            d_send, d_pos = [], []
            for r in range(k):
                ids = torch.from_numpy(routing[r].astype(np.int32)).cuda()
                x = to_device(xs[r], "bfloat16")
                send, _, pos_of, cnt = _pack_on_device(ids, x, experts, k, s)
                d_counts[r].copy_(cnt)
                d_send.append(send.view(-1))
                d_pos.append(pos_of)
            w_dev = [torch.from_numpy(ws[r]).cuda() for r in range(k)]   # no pageable copy while the stream is held
            cap = [int(counts[:, d].sum()) + 4096 for d in range(k)]
            d_recv = [torch.empty(cap[d], dtype=torch.bfloat16, device="cuda") for d in range(k)]
            d_back = [torch.empty_like(t) for t in d_send]
        c.alltoall_device_counts(d_send, d_recv, d_counts, cap, hoc.BFLOAT16, stream=s)
        c.alltoall_device_counts(d_recv, d_back, d_counts, [t.numel() for t in d_back], hoc.BFLOAT16, stream=s,
                                 transpose=True)
        ys = []
        with torch.cuda.stream(s):
            for r in range(k):
                y = torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda")
                hoc.ep_combine(d_back[r], d_pos[r], w_dev[r], tokens, topk, hidden, y, stream=s)
                ys.append(y)
        c.wait(s, timeout_ms=60000)
        for r in range(k):
            assert np.array_equal(to_host(ys[r], "bfloat16"), want_y[r]), r
        assert c.proxy_status()["completed"] == 2


@pytest.mark.parametrize("hidden", [1, 8])   # the scalar combine, and the vector combine with the value in every lane
def test_combine_golden_cases(hidden):
    """The hand-derived combine cases straight from the golden file (no oracle)."""
    from tests import pins
    for c in pins.load_ep_combine_cases():
        tokens = len(c["y"])
        packed = np.zeros((tokens * c["topk"], hidden), dtype=np.uint16)  # the API's [tokens*topk, hidden] rows
        packed[: len(c["rows"])] = np.repeat(c["rows"], hidden, axis=1)
        rows = torch.from_numpy(packed.view(np.int16).copy()).cuda().view(torch.bfloat16)
        pos = torch.from_numpy(c["pos_of"].astype(np.int32)).cuda()
        w = torch.from_numpy(c["weights"].copy()).cuda()
        y = torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda")
        hoc.ep_combine(rows, pos, w, tokens, c["topk"], hidden, y)
        torch.cuda.synchronize()
        got = y.view(torch.int16).cpu().numpy().astype(np.int64) & 0xFFFF
        assert np.array_equal(got, np.repeat(c["y"].astype(np.int64)[:, None], hidden, axis=1)), \
            (c["name"], hidden, [hex(int(v)) for v in got.reshape(-1)])


# scalar; one vector per lane; one slice and a 16-byte tail (1 KiB slices at topk 4, 2 KiB at 2-3);
# rows of 4112 B: several whole slices and a 16-byte tail
@pytest.mark.parametrize("hidden", [1, 8, 520, 2056])
@pytest.mark.parametrize("engine", [None, "lsu"])   # TMA-fed combine (default), vector-load combine
def test_fused_combine_golden_cases(hidden, engine, monkeypatch):
    """The hand-derived combine cases through the combine that reads the rows in place: one rank,
    one expert, every row where the case puts it."""
    from tests import pins
    if engine:
        monkeypatch.setenv("HOC_EP_COMBINE", engine)
    for c in pins.load_ep_combine_cases():
        tokens, topk = len(c["y"]), c["topk"]
        n_rows = len(c["rows"])
        cap = (n_rows + 2) * hidden
        rows = np.zeros((n_rows + 2, hidden), dtype=np.uint16)
        rows[:n_rows] = np.repeat(c["rows"], hidden, axis=1)
        recv = torch.from_numpy(rows.view(np.int16).reshape(-1).copy()).cuda().view(torch.bfloat16)
        ids = torch.zeros(tokens * topk, dtype=torch.int32, device="cuda")
        pos = torch.from_numpy(c["pos_of"].astype(np.int32)).cuda()
        counts = torch.tensor([[n_rows * hidden]], dtype=torch.int64, device="cuda")
        w = torch.from_numpy(c["weights"].copy()).cuda()
        y = torch.full((tokens, hidden), 7.0, dtype=torch.bfloat16, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        hoc.ep_combine_fused([recv], [cap], [ids], [pos], counts, [w], tokens, topk, hidden, 1, [y], status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, c["name"]
        got = y.view(torch.int16).cpu().numpy().astype(np.int64) & 0xFFFF
        assert np.array_equal(got, np.repeat(c["y"].astype(np.int64)[:, None], hidden, axis=1)), \
            (c["name"], hidden, engine, [hex(int(v)) for v in got.reshape(-1)[:16]])


# ---------------------------------------------------------------- fused with the exchange
def _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden):
    """pack -> all-to-all -> (identity experts) -> inverse all-to-all -> combine, on the CPU."""
    packs = [o_ep.pack(xs[r], routing[r], experts, k) for r in range(k)]
    counts = np.stack([p[3] for p in packs])
    recv = o_a2a.alltoallv([p[0].reshape(-1) for p in packs], counts)
    back = o_a2a.alltoallv(recv, o_a2a.transpose_counts(counts))
    ys = [o_ep.combine(back[r].reshape(-1, hidden), packs[r][2], ws[r], topk) for r in range(k)]
    return packs, counts, recv, ys


def _fused_on_device(k, xs, routing, ws, experts, topk, caps, recv_offset=0, y_offset=0):
    from tests.gpu_util import Guarded
    tokens, hidden = xs[0].shape
    n = tokens * topk
    d_ids = [torch.from_numpy(np.ascontiguousarray(r, dtype=np.int32).reshape(-1)).cuda() for r in routing]
    d_x = [to_device(x, "bfloat16") for x in xs]
    recv = [Guarded(max(1, c), "bfloat16", offset_elems=recv_offset) for c in caps]
    pos = [torch.full((max(1, n),), -7, dtype=torch.int32, device="cuda") for _ in range(k)]
    counts = torch.full((k, k), -1, dtype=torch.int64, device="cuda")
    wsp = torch.empty(max(1, k * hoc.ep_pack_workspace(tokens, topk, experts)), dtype=torch.int32, device="cuda")
    status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    hoc.ep_dispatch_fused(d_ids, d_x, experts, [g.tensor for g in recv], caps, pos, counts, wsp, status)
    w = [torch.from_numpy(x).cuda() for x in ws]
    ys = [Guarded(tokens * hidden, "bfloat16", offset_elems=y_offset) for _ in range(k)]
    hoc.ep_combine_fused([g.tensor for g in recv], caps, d_ids, pos, counts, w, tokens, topk, hidden, experts,
                         [g.tensor for g in ys], status)
    torch.cuda.synchronize()
    return recv, pos, counts, status, ys


@pytest.mark.parametrize("k,tokens,hidden,drop,experts,topk,recv_offset", [
    (8, 4096, 2048, False, 64, 6, 0),   # the EP workload's shape
    (8, 333, 40, True, 64, 6, 0),       # partial tile, dropped pairs; rows of 80 B: one partial slice each
    (8, 250, 36, True, 64, 6, 0),       # rows of 72 B: byte dispatch, scalar combine
    (8, 5000, 64, True, 96, 4, 0),      # ragged last tile, 12 experts per rank
    (3, 1000, 64, True, 48, 4, 0),      # three ranks
    (8, 700, 16, False, 2048, 2, 0),    # more than 1024 experts: the one-CTA-per-expert sort
    (8, 200, 24, False, 64, 10, 0),     # topk above the batched loads: the one-load-at-a-time combine
    (8, 100, 16, True, 64, 40, 0),      # topk above a warp
    (8, 777, 64, True, 64, 6, 1),       # receive buffers 2 bytes off alignment: byte dispatch, scalar combine
    (1, 300, 64, True, 8, 3, 0),        # one rank: everything stays home
    (4, 300, 4100, True, 32, 1, 0),     # top-1: 4 KiB combine slices, rows of 8200 B (two whole, one ragged)
    (4, 300, 2100, True, 32, 2, 0),     # top-2: 2 KiB combine slices, rows of 4200 B
])
@pytest.mark.parametrize("engines", [None, ("bulk", "lsu")])
def test_fused_dispatch_and_combine_match_oracle(k, tokens, hidden, drop, experts, topk, recv_offset, engines,
                                                 monkeypatch):
    if engines:   # the other engines: TMA bulk-copy dispatch, vector-load combine
        monkeypatch.setenv("HOC_EP_DISPATCH", engines[0])
        monkeypatch.setenv("HOC_EP_COMBINE", engines[1])
    routing = [r.copy() for r in inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5200 + k)]
    if drop:
        routing[0][3 % tokens, 0] = -5
        routing[k - 1][7 % tokens, topk - 1] = experts
    xs = [inputs.normal_bf16(tokens * hidden, 5700 + r).reshape(tokens, hidden) for r in range(k)]
    rng = np.random.default_rng(5800 + k)
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) + 3 * hidden for d in range(k)]     # room to spare: the guard must stay
    recv, pos, d_counts, status, ys = _fused_on_device(k, xs, routing, ws, experts, topk, caps, recv_offset)
    assert int(status.item()) == 0
    assert np.array_equal(d_counts.cpu().numpy(), counts)
    for r in range(k):
        assert np.array_equal(pos[r].cpu().numpy()[: tokens * topk], packs[r][2]), r
    for d in range(k):
        got = recv[d].host()
        n = len(want_recv[d])
        assert np.array_equal(got[:n], want_recv[d]), f"dispatch rank {d}"
        assert np.all(got[n:] == 0xA5A5), f"rank {d}: written past its rows"
        recv[d].check()
    for r in range(k):
        ys[r].check()
        assert np.array_equal(ys[r].host().reshape(tokens, hidden), want_y[r]), f"combine rank {r}"


def test_fused_dispatch_reports_rows_that_do_not_fit():
    k, tokens, hidden, experts, topk = 4, 300, 64, 32, 4
    routing = inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5300)
    xs = [inputs.normal_bf16(tokens * hidden, 5900 + r).reshape(tokens, hidden) for r in range(k)]
    ws = [np.ones(tokens * topk, np.float32) for _ in range(k)]
    packs, counts, want_recv, _ = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    need = [int(counts[:, d].sum()) for d in range(k)]
    caps = list(need)
    caps[0] = need[0] - 5 * hidden                                      # rank 0 lacks room for five rows
    recv, _, _, status, _ = _fused_on_device(k, xs, routing, ws, experts, topk, caps)
    st = int(status.item())
    assert st & 1 and st & 2                                            # dispatch and combine both saw it
    for d in range(k):
        recv[d].check()                                                 # nothing written outside a buffer
        if d:
            assert np.array_equal(recv[d].host(), want_recv[d])         # the other ranks are complete
    assert np.array_equal(recv[0].host(), want_recv[0][: caps[0]])      # rank 0 holds the rows that fit


def test_fused_zero_tokens():
    k, hidden, experts = 4, 64, 16
    ids = [torch.empty(0, dtype=torch.int32, device="cuda") for _ in range(k)]
    xs = [torch.empty((0, hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    recv = [torch.empty(hidden, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    counts = torch.full((k, k), 5, dtype=torch.int64, device="cuda")
    status = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    ws = torch.empty(1, dtype=torch.int32, device="cuda")
    hoc.ep_dispatch_fused(ids, xs, experts, recv, [hidden] * k, ids, counts, ws, status)
    torch.cuda.synchronize()
    assert counts.abs().sum().item() == 0 and int(status.item()) == 0


@pytest.mark.parametrize("engines", [None, ("bulk", "lsu")])
def test_fused_sixteen_ranks_and_misaligned_outputs(engines, monkeypatch):
    # the most ranks a call takes, and outputs 2 bytes off alignment (vector dispatch, scalar combine)
    if engines:
        monkeypatch.setenv("HOC_EP_DISPATCH", engines[0])
        monkeypatch.setenv("HOC_EP_COMBINE", engines[1])
    k, tokens, hidden, experts, topk = 16, 300, 128, 64, 4
    routing = [r.copy() for r in inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5400)]
    xs = [inputs.normal_bf16(tokens * hidden, 6000 + r).reshape(tokens, hidden) for r in range(k)]
    rng = np.random.default_rng(6100)
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) for d in range(k)]
    for y_offset in (0, 1):
        recv, pos, d_counts, status, ys = _fused_on_device(k, xs, routing, ws, experts, topk, caps, 0, y_offset)
        assert int(status.item()) == 0
        for d in range(k):
            assert np.array_equal(recv[d].host(), want_recv[d]), d
        for r in range(k):
            ys[r].check()
            assert np.array_equal(ys[r].host().reshape(tokens, hidden), want_y[r]), (y_offset, r)


def test_fused_combine_reports_rows_outside_its_buffers():
    # the dispatch fits; the combine is told a smaller buffer for rank 0: the rows past it add nothing,
    # bit 1 of the status is set, and nothing is written outside the outputs
    from tests.gpu_util import Guarded
    k, tokens, hidden, experts, topk = 4, 200, 64, 16, 3
    routing = inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5500)
    xs = [inputs.normal_bf16(tokens * hidden, 6200 + r).reshape(tokens, hidden) for r in range(k)]
    ws = [np.ones(tokens * topk, np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) for d in range(k)]
    d_ids = [torch.from_numpy(np.ascontiguousarray(r, dtype=np.int32).reshape(-1)).cuda() for r in routing]
    d_x = [to_device(x, "bfloat16") for x in xs]
    recv = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for c in caps]
    pos = [torch.empty(tokens * topk, dtype=torch.int32, device="cuda") for _ in range(k)]
    d_counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    hoc.ep_dispatch_fused(d_ids, d_x, experts, recv, caps, pos, d_counts, wsp, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    small = list(caps)
    small[0] = caps[0] - 4 * hidden
    ys = [Guarded(tokens * hidden, "bfloat16") for _ in range(k)]
    w = [torch.from_numpy(x).cuda() for x in ws]
    hoc.ep_combine_fused(recv, small, d_ids, pos, d_counts, w, tokens, topk, hidden, experts, [g.tensor for g in ys],
                         status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    for r in range(k):
        ys[r].check()


@pytest.mark.parametrize("engines", [None, ("bulk", "lsu")])
@pytest.mark.parametrize("k,tokens,hidden,experts,topk", [(8, 4096, 2048, 64, 6), (3, 500, 36, 48, 4),
                                                          (8, 300, 64, 2048, 2), (4, 300, 4100, 32, 1)])
def test_pack_all_and_combine_all_match_oracle(k, tokens, hidden, experts, topk, engines, monkeypatch):
    # every rank's pack in one pass, the two copy-engine exchanges, every rank's combine in one pass
    if engines:
        monkeypatch.setenv("HOC_EP_DISPATCH", engines[0])
        monkeypatch.setenv("HOC_EP_COMBINE", engines[1])
    from tests.gpu_util import Guarded
    routing = [r.copy() for r in inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=5600 + k)]
    routing[0][1, 0] = -1
    xs = [inputs.normal_bf16(tokens * hidden, 6300 + r).reshape(tokens, hidden) for r in range(k)]
    rng = np.random.default_rng(6400)
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    n = tokens * topk
    d_ids = [torch.from_numpy(np.ascontiguousarray(r, dtype=np.int32).reshape(-1)).cuda() for r in routing]
    d_x = [to_device(x, "bfloat16") for x in xs]
    send = [Guarded(n * hidden, "bfloat16") for _ in range(k)]
    pos = [torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(k)]
    d_counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    status = torch.full((1,), 9, dtype=torch.int32, device="cuda")
    hoc.ep_pack_all(d_ids, d_x, experts, [g.tensor for g in send], [n * hidden] * k, pos, d_counts, wsp, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(d_counts.cpu().numpy(), counts)
    for r in range(k):
        nv = len(packs[r][1])
        assert np.array_equal(send[r].host()[: nv * hidden], packs[r][0].reshape(-1)), r
        assert np.all(send[r].host()[nv * hidden:] == 0xA5A5), r      # nothing past the valid rows
        assert np.array_equal(pos[r].cpu().numpy(), packs[r][2]), r
        send[r].check()
    caps = [int(counts[:, d].sum()) for d in range(k)]
    with hoc.Comm(k, 0) as c:
        recv = [torch.empty(max(1, v), dtype=torch.bfloat16, device="cuda") for v in caps]
        back = [torch.empty(n * hidden, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
        c.alltoall([g.tensor for g in send], recv, sendcounts=counts, dtype=hoc.BFLOAT16)
        c.alltoall(recv, back, sendcounts=counts.T.copy(), dtype=hoc.BFLOAT16)
        c.wait()
    ys = [Guarded(tokens * hidden, "bfloat16") for _ in range(k)]
    w = [torch.from_numpy(x).cuda() for x in ws]
    hoc.ep_combine_all(back, [n * hidden] * k, pos, w, tokens, topk, hidden, [g.tensor for g in ys], status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for r in range(k):
        ys[r].check()
        assert np.array_equal(ys[r].host().reshape(tokens, hidden), want_y[r]), r


@pytest.mark.parametrize("seed", range(6))
def test_fused_and_all_rank_paths_on_random_shapes(seed, monkeypatch):
    """Random rank counts, token counts, row widths, expert counts, topk, dropped pairs and buffer
    offsets; both engine sets; the fused path and the all-rank pack / combine against the oracle."""
    rng = np.random.default_rng(9100 + seed)
    k = int(rng.choice([1, 2, 3, 5, 8, 16]))
    per = int(rng.integers(1, 9))
    experts = k * per
    topk = int(rng.integers(1, min(experts, 12) + 1))
    tokens = int(rng.integers(1, 700))
    hidden = int(rng.choice([8, 16, 24, 40, 64, 72, 136, 520]))
    if seed % 2:
        monkeypatch.setenv("HOC_EP_DISPATCH", "bulk")
        monkeypatch.setenv("HOC_EP_COMBINE", "lsu")
    routing = [np.stack([rng.permutation(experts)[:topk] for _ in range(tokens)]) for _ in range(k)]
    for r in range(k):                                   # a few dropped pairs
        for _ in range(int(rng.integers(0, 4))):
            routing[r][int(rng.integers(tokens)), int(rng.integers(topk))] = int(rng.choice([-1, experts, -7]))
    xs = [inputs.normal_bf16(tokens * hidden, 9200 + 17 * seed + r).reshape(tokens, hidden) for r in range(k)]
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) + int(rng.integers(0, 3)) * hidden for d in range(k)]
    off = int(rng.integers(0, 2))
    recv, pos, d_counts, status, ys = _fused_on_device(k, xs, routing, ws, experts, topk, caps, off, off)
    assert int(status.item()) == 0, (seed, k, tokens, hidden, experts, topk)
    assert np.array_equal(d_counts.cpu().numpy(), counts)
    for d in range(k):
        recv[d].check()
        assert np.array_equal(recv[d].host()[: len(want_recv[d])], want_recv[d]), (seed, d)
    for r in range(k):
        ys[r].check()
        assert np.array_equal(ys[r].host().reshape(tokens, hidden), want_y[r]), (seed, r)
    # the all-rank pack and combine, with the oracle's exchange in between
    n = tokens * topk
    d_ids = [torch.from_numpy(np.ascontiguousarray(rr, dtype=np.int32).reshape(-1)).cuda() for rr in routing]
    d_x = [to_device(x, "bfloat16") for x in xs]
    send = [torch.empty(max(1, n * hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    pos2 = [torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(k)]
    c2 = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    hoc.ep_pack_all(d_ids, d_x, experts, send, [n * hidden] * k, pos2, c2, wsp, st)
    torch.cuda.synchronize()
    back_host = o_a2a.alltoallv(o_a2a.alltoallv([to_host(send[r], "bfloat16")[: len(packs[r][1]) * hidden]
                                                 for r in range(k)], counts), o_a2a.transpose_counts(counts))
    back = [to_device(np.concatenate([b_, np.zeros(n * hidden - len(b_), np.uint16)]) if n * hidden else
                      np.zeros(1, np.uint16), "bfloat16") for b_ in back_host]
    y2 = [torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    hoc.ep_combine_all(back, [max(1, n * hidden)] * k, pos2, [torch.from_numpy(w).cuda() for w in ws], tokens, topk,
                       hidden, y2, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for r in range(k):
        assert np.array_equal(to_host(y2[r], "bfloat16").reshape(tokens, hidden), want_y[r]), (seed, r)


def test_fused_round_trip_replays_from_a_cuda_graph():
    """The fused dispatch and combine captured once into a CUDA graph, then replayed on other
    routings and rows copied into the captured buffers: every replay matches the oracle of its
    own inputs (the sort, the counts and every row position are recomputed on the device)."""
    k, tokens, hidden, experts, topk = 8, 512, 256, 64, 6
    cases = []
    for seed in (0, 1, 2):
        routing = [r.copy() for r in inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=7000 + 100 * seed)]
        if seed == 2:
            routing[3][5, 2] = -1                       # a dropped pair
        xs = [inputs.normal_bf16(tokens * hidden, 7300 + 100 * seed + r).reshape(tokens, hidden) for r in range(k)]
        rng = np.random.default_rng(7600 + seed)
        ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
        cases.append((routing, xs, ws, _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)[3]))
    cap = k * tokens * topk * hidden                    # room for any routing
    d_ids = [torch.empty(tokens * topk, dtype=torch.int32, device="cuda") for _ in range(k)]
    d_x = [torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    d_w = [torch.empty(tokens * topk, dtype=torch.float32, device="cuda") for _ in range(k)]
    recv = [torch.empty(cap, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    pos = [torch.empty(tokens * topk, dtype=torch.int32, device="cuda") for _ in range(k)]
    counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    ys = [torch.empty((tokens, hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    s = torch.cuda.Stream()

    def load(case):
        routing, xs, ws, _ = case
        for r in range(k):
            d_ids[r].copy_(torch.from_numpy(np.ascontiguousarray(routing[r], dtype=np.int32).reshape(-1)))
            d_x[r].copy_(to_device(xs[r], "bfloat16"))
            d_w[r].copy_(torch.from_numpy(ws[r]))
        torch.cuda.synchronize()

    def round_trip():
        hoc.ep_dispatch_fused(d_ids, d_x, experts, recv, [cap] * k, pos, counts, wsp, status, stream=s)
        hoc.ep_combine_fused(recv, [cap] * k, d_ids, pos, counts, d_w, tokens, topk, hidden, experts, ys, status,
                             stream=s)

    load(cases[0])
    with torch.cuda.stream(s):
        round_trip()                                    # first calls outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        round_trip()
    for case in (cases[1], cases[2], cases[0]):
        load(case)
        for y in ys:
            y.fill_(7.0)
        status.fill_(99)                                # the graph clears it
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for r in range(k):
            assert np.array_equal(to_host(ys[r], "bfloat16").reshape(tokens, hidden), case[3][r]), r
    # the all-rank pack and combine, with the rows left in place between them (the two exchanges of
    # the round trip bring every row back where the pack put it): the same results
    send = [torch.empty(tokens * topk * hidden, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    scap = [tokens * topk * hidden] * k

    def pack_combine():
        hoc.ep_pack_all(d_ids, d_x, experts, send, scap, pos, counts, wsp, status, stream=s)
        hoc.ep_combine_all(send, scap, pos, d_w, tokens, topk, hidden, ys, status, stream=s)

    load(cases[0])
    with torch.cuda.stream(s):
        pack_combine()
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        pack_combine()
    for case in (cases[2], cases[1]):
        load(case)
        for y in ys:
            y.fill_(7.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g2.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for r in range(k):
            assert np.array_equal(to_host(ys[r], "bfloat16").reshape(tokens, hidden), case[3][r]), r


@pytest.mark.parametrize("stage", ["dispatch", "combine"])
def test_bulk_copy_waits_give_up_into_the_status_word(stage, monkeypatch):
    """HOC_FAULT=ep_stall (injected on the host): every mbarrier of the TMA bulk-copy dispatch or
    combine expects 16 bytes more than its loads bring, so no wait completes; each gives up after
    its 0.1 s limit, sets status bit 2 and drains its own loads, and the next call is exact."""
    k, tokens, hidden, experts, topk = 4, 300, 64, 32, 4
    routing = inputs.ep_routing(k, tokens, experts, topk, 1.1, seed_base=7900)
    xs = [inputs.normal_bf16(tokens * hidden, 7950 + r).reshape(tokens, hidden) for r in range(k)]
    rng = np.random.default_rng(7990)
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) for d in range(k)]
    monkeypatch.setenv("HOC_EP_DISPATCH", "bulk")      # the dispatch's bulk-copy engine (the combine's is the default)
    d_ids = [torch.from_numpy(np.ascontiguousarray(r, dtype=np.int32).reshape(-1)).cuda() for r in routing]
    d_x = [to_device(x, "bfloat16") for x in xs]
    d_w = [torch.from_numpy(x).cuda() for x in ws]
    recv = [torch.zeros(c, dtype=torch.bfloat16, device="cuda") for c in caps]
    pos = [torch.empty(tokens * topk, dtype=torch.int32, device="cuda") for _ in range(k)]
    d_counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    ys = [torch.zeros((tokens, hidden), dtype=torch.bfloat16, device="cuda") for _ in range(k)]

    def dispatch(status):
        hoc.ep_dispatch_fused(d_ids, d_x, experts, recv, caps, pos, d_counts, wsp, status)

    def combine(status):
        hoc.ep_combine_fused(recv, caps, d_ids, pos, d_counts, d_w, tokens, topk, hidden, experts, ys, status)

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if stage == "dispatch":
        monkeypatch.setenv("HOC_FAULT", "ep_stall")
        dispatch(status)
    else:
        dispatch(status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        monkeypatch.setenv("HOC_FAULT", "ep_stall")
        combine(status)
    torch.cuda.synchronize()
    assert int(status.item()) & 4, int(status.item())
    monkeypatch.delenv("HOC_FAULT")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dispatch(status)
    combine(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for d in range(k):
        assert np.array_equal(to_host(recv[d], "bfloat16"), want_recv[d]), d
    for r in range(k):
        assert np.array_equal(to_host(ys[r], "bfloat16").reshape(tokens, hidden), want_y[r]), r


def test_fused_dispatch_past_the_grid_cap():
    """More (source, token) work items than the dispatch grid's 2^20 CTAs x 8 warps: 8 ranks x
    1,100,000 tokens of 6-byte rows (the byte path, one warp per token), so warps loop over
    several items; results against the oracle."""
    k, tokens, hidden, experts, topk = 8, 1_100_000, 3, 16, 1
    assert k * tokens > (1 << 20) * 8
    rng = np.random.default_rng(9900)
    routing = [rng.integers(0, experts, size=(tokens, topk)) for _ in range(k)]
    routing[2][17, 0] = -1                                   # a dropped pair
    xs = [inputs.normal_bf16(tokens * hidden, 9910 + r).reshape(tokens, hidden) for r in range(k)]
    ws = [rng.random(tokens * topk).astype(np.float32) for _ in range(k)]
    packs, counts, want_recv, want_y = _oracle_round_trip(xs, routing, ws, experts, k, topk, hidden)
    caps = [int(counts[:, d].sum()) for d in range(k)]
    recv, pos, d_counts, status, ys = _fused_on_device(k, xs, routing, ws, experts, topk, caps)
    assert int(status.item()) == 0
    assert np.array_equal(d_counts.cpu().numpy(), counts)
    for d in range(k):
        assert np.array_equal(recv[d].host()[: len(want_recv[d])], want_recv[d]), d
        recv[d].check()
    for r in range(k):
        assert np.array_equal(ys[r].host().reshape(tokens, hidden), want_y[r]), r
