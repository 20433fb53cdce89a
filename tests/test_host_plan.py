"""Host logic on CPU: the scheduler's plans (via hoc_plan_query), the C ABI
exports, and host-side fault injection.  No GPU needed."""
import os
import re
from collections import defaultdict

import numpy as np
import pytest

from collective_communication_schedules_gb300 import hoc
from oracle import ring as o_ring

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from collective_communication_schedules_gb300 import build
    build.build()


def _cover(intervals):
    """Sorted, merged coverage of byte intervals and whether any overlapped."""
    iv = sorted(intervals)
    overlap = any(iv[i][1] > iv[i + 1][0] for i in range(len(iv) - 1))
    return iv, overlap


def _total(iv):
    return sum(b - a for a, b in iv)


# ------------------------------------------------------------------ exports
def test_every_declared_symbol_is_exported():
    lib = hoc.lib()
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^\s*(?:hocResult_t|const char\*)\s+(hoc_\w+)\s*\(", text, re.M))
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n
    assert set(hoc._SIGS) <= names


def _prototypes():
    """name -> list of parameter declarations of every function the headers declare."""
    protos = {}
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:hocResult_t|const char\s*\*)\s+(hoc_\w+)\s*\(([^;]*?)\)\s*;", text, re.M | re.S):
            params = " ".join(m.group(2).split())
            protos[m.group(1)] = [] if params in ("", "void") else [q.strip() for q in params.split(",")]
    return protos


def test_binding_signatures_match_the_headers():
    """Each ctypes entry has the header's parameter count, pointer-ness and integer widths."""
    import ctypes as C
    protos = _prototypes()
    for name, (res, args) in hoc._SIGS.items():
        params = protos[name]
        assert len(args) == len(params), (name, len(args), params)
        for a, q in zip(args, params):
            is_ptr = "*" in q or q.split()[0] == "hocComm_t"   # hocComm_t is a pointer typedef
            ctype_ptr = a in (C.c_void_p, C.c_char_p) or (isinstance(a, type) and issubclass(a, C._Pointer))
            assert is_ptr == ctype_ptr, (name, q, a)
            if not is_ptr:
                want = {"size_t": C.c_size_t, "uint64_t": C.c_uint64, "uint16_t": C.c_uint16}
                base = q.split()[0]
                if base in want:
                    assert C.sizeof(a) == C.sizeof(want[base]), (name, q, a)
                elif base in ("int", "hocDataType_t", "hocRedOp_t", "hocResult_t", "hocKernel_t"):
                    assert C.sizeof(a) == C.sizeof(C.c_int), (name, q, a)
                else:
                    raise AssertionError(f"{name}: unchecked parameter type {q!r}")


def test_no_device_is_a_clean_error():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(hoc.HocError) as e:
        hoc.Comm(4)
    assert e.value.code == hoc.ERR_NO_DEVICE
    with pytest.raises(hoc.HocError):
        hoc.sm_count()


# ---------------------------------------------------------------- allreduce
@pytest.mark.parametrize("path", ["ce", "tma"])
@pytest.mark.parametrize("k,n,chunk", [(4, 1 << 20, 1 << 18), (8, 1000003, 1 << 16), (3, 17, 256), (5, 4096 * 5 + 3, 4096),
                                       (6, 300007, 1 << 14), (7, 50000, 0)])
def test_allreduce_plan_covers_every_block_once(path, k, n, chunk):
    b = 4
    items = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.FLOAT32, config=hoc.Config(path=path, chunk_bytes=chunk))
    sizes, offs = o_ring.block_partition(n, k)
    red = defaultdict(list)
    moves = defaultdict(list)
    steps = {}
    for it in items:
        steps.setdefault(it["step"], it)
        if it["kind"] == hoc.ITEM_REDUCE:
            assert it["stream"] == 0
            red[it["dst_rank"]].append((it["src_off"], it["src_off"] + it["bytes"]))
            assert it["src_off"] == it["dst_off"]
        else:
            assert it["kind"] == (hoc.ITEM_TMA if path == "tma" else hoc.ITEM_COPY)
            assert it["src_buf"] == hoc.BUF_RECV and it["dst_buf"] == hoc.BUF_RECV
            assert it["src_off"] == it["dst_off"] and it["src_rank"] != it["dst_rank"]
            moves[(it["src_rank"], it["dst_rank"])].append((it["src_off"], it["src_off"] + it["bytes"]))
            # the move waits for the reduce step of its own chunk
            w = steps[it["wait0"]]
            assert it["n_waits"] >= 1 and w["kind"] == hoc.ITEM_REDUCE and w["stage"] == it["stage"]
    for r in range(k):
        iv, ov = _cover(red[r])
        assert not ov and _total(iv) == sizes[r] * b
        assert iv[0][0] == offs[r] * b and iv[-1][1] == (offs[r] + sizes[r]) * b
        for d in range(k):
            if d == r:
                continue
            iv, ov = _cover(moves[(r, d)])
            assert not ov and _total(iv) == sizes[r] * b
            assert iv[0][0] == offs[r] * b


@pytest.mark.parametrize("path", ["ce", "tma"])
def test_allreduce_chunk_boundaries_sit_on_4_kib_offsets(path):
    """Blocks that start off a 4 KiB boundary (k = 6, 2^27 bf16): every chunk of a block but its first starts
    on one, the first runs from the block's start to one chunk past the block's first boundary, and the
    blocks (which rank folds what) are the oracle's."""
    k, n, b = 6, 1 << 27, 2
    items = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.BFLOAT16, config=hoc.Config(path=path))
    sizes, offs = o_ring.block_partition(n, k)
    assert any((offs[r] * b) % 4096 for r in range(k))
    for r in range(k):
        segs = sorted((it["src_off"], it["bytes"]) for it in items
                      if it["kind"] == hoc.ITEM_REDUCE and it["dst_rank"] == r)
        assert segs[0][0] == offs[r] * b
        assert all(off % 4096 == 0 for off, _ in segs[1:])
        assert sum(nb for _, nb in segs) == sizes[r] * b
        ce = segs[1][1]
        assert segs[0][0] + segs[0][1] == -(-offs[r] * b // 4096) * 4096 + ce
    # a chunk size that is not a whole number of 4 KiB units is cut down to one (k = 12: 32 MiB / 12)
    items = hoc.plan_query(12, hoc.OP_ALLREDUCE, n, hoc.BFLOAT16, config=hoc.Config(path=path))
    offs12 = [it["src_off"] for it in items if it["kind"] == hoc.ITEM_REDUCE]
    sizes12, starts12 = o_ring.block_partition(n, 12)
    assert all(o % 4096 == 0 for o in offs12 if o not in {s * b for s in starts12})


@pytest.mark.parametrize("op", ["allgather", "alltoall"])
def test_move_pieces_start_on_4_kib_destination_offsets(op):
    """Copy-engine moves whose destinations start off a 4 KiB boundary: each move's pieces cover it once,
    every piece but the first starts on a 4 KiB destination offset, and no piece is left under a quarter
    chunk unless the whole move is."""
    k, chunk, b = 4, 4 << 20, 2
    cfg = hoc.Config(path="ce", chunk_bytes=chunk)
    if op == "allgather":
        count = (9 << 20) // b + 8                          # blocks of 9 MiB + 16 B: destinations r * that
        items = hoc.plan_query(k, hoc.OP_ALLGATHER, count, hoc.BFLOAT16, config=cfg)
    else:
        counts = np.full((k, k), (9 << 20) // b + 8, dtype=np.uint64)
        counts[1, 2] = 3                                    # a flow far under a quarter chunk
        items = hoc.plan_query(k, hoc.OP_ALLTOALL, 0, hoc.BFLOAT16, counts=counts, config=cfg)
    moves = defaultdict(list)
    for it in items:
        if it["kind"] == hoc.ITEM_COPY:
            moves[(it["src_rank"], it["dst_rank"])].append((it["dst_off"], it["src_off"], it["bytes"]))
    assert moves
    for key, ps in moves.items():
        ps.sort()
        total = sum(p[2] for p in ps)
        for (d0, s0, n0), (d1, s1, n1) in zip(ps, ps[1:]):
            assert d0 + n0 == d1 and s0 + n0 == s1, key           # contiguous on both sides
        for d, _, n in ps[1:]:
            assert d % 4096 == 0, key
        assert all(n >= chunk // 4 for _, _, n in ps) or len(ps) == 1, key
        assert total == (3 * b if (op, key) == ("alltoall", (1, 2)) else ((9 << 20) // b + 8) * b), key


def test_allreduce_chunking_and_striping():
    k, n = 8, 134_217_728
    cfg = hoc.Config(path="ce", chunk_bytes=4 << 20, n_copy_streams=4)
    items = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.BFLOAT16, config=cfg)
    reduce_steps = {it["step"] for it in items if it["kind"] == hoc.ITEM_REDUCE}
    assert len(reduce_steps) == (n // k * 2) // (4 << 20)           # 32 MiB blocks / 4 MiB chunks
    streams = {it["stream"] for it in items if it["kind"] == hoc.ITEM_COPY}
    assert streams == {1, 2, 3, 4}
    per_stream = defaultdict(int)
    for it in items:
        if it["kind"] == hoc.ITEM_COPY:
            per_stream[it["stream"]] += it["bytes"]
    assert max(per_stream.values()) == min(per_stream.values())      # even striping


def test_fused_allreduce_is_one_launch():
    items = hoc.plan_query(8, hoc.OP_ALLREDUCE, 1001, hoc.BFLOAT16, config=hoc.Config(path="fused"))
    assert {it["kind"] for it in items} == {hoc.ITEM_FUSED}
    assert len({it["step"] for it in items}) == 1 and len(items) == 8
    auto = hoc.plan_query(8, hoc.OP_ALLREDUCE, 1001, hoc.BFLOAT16, config=hoc.Config(path="auto"))
    assert auto == items


def test_auto_allreduce_under_an_sm_budget_moves_on_copy_engines():
    # with the whole GPU AUTO fuses; with an SM budget the few SMs only reduce
    budget = hoc.plan_query(8, hoc.OP_ALLREDUCE, 1 << 20, hoc.BFLOAT16,
                            config=hoc.Config(path="auto", reduce_max_sms=8))
    ce = hoc.plan_query(8, hoc.OP_ALLREDUCE, 1 << 20, hoc.BFLOAT16, config=hoc.Config(path="ce", reduce_max_sms=8))
    assert budget == ce
    assert {it["kind"] for it in budget} == {hoc.ITEM_REDUCE, hoc.ITEM_COPY}


def test_pipeline_depth_adds_backpressure_edges():
    cfg = hoc.Config(path="ce", chunk_bytes=1 << 16, pipeline_depth=2)
    items = hoc.plan_query(4, hoc.OP_ALLREDUCE, 1 << 20, hoc.FLOAT32, config=cfg)
    by_step = {}
    for it in items:
        by_step.setdefault(it["step"], it)
    reds = sorted((it for it in by_step.values() if it["kind"] == hoc.ITEM_REDUCE), key=lambda x: x["stage"])
    assert reds[0]["n_waits"] == 0 and reds[1]["n_waits"] == 0
    for r in reds[2:]:
        w = by_step[r["wait0"]]
        assert w["kind"] == hoc.ITEM_COPY and w["stage"] == r["stage"] - 2


def test_reduce_scatter_plan():
    k, rc = 8, 1_638_400
    items = hoc.plan_query(k, hoc.OP_REDUCE_SCATTER, rc, hoc.BFLOAT16)
    assert len(items) == k and all(it["kind"] == hoc.ITEM_REDUCE for it in items)
    for it in items:
        r = it["dst_rank"]
        assert it["src_off"] == r * rc * 2 and it["dst_off"] == 0 and it["bytes"] == rc * 2


# ---------------------------------------------------------------- allgather
@pytest.mark.parametrize("path", ["ce", "tma"])
def test_allgather_plan_covers_every_pair(path):
    k, sc = 5, 300001
    items = hoc.plan_query(k, hoc.OP_ALLGATHER, sc, hoc.BFLOAT16, config=hoc.Config(path=path, chunk_bytes=1 << 16))
    got = defaultdict(list)
    for it in items:
        assert it["src_buf"] == hoc.BUF_SEND and it["dst_buf"] == hoc.BUF_RECV
        assert it["dst_off"] - it["src_off"] == it["src_rank"] * sc * 2
        got[(it["src_rank"], it["dst_rank"])].append((it["src_off"], it["src_off"] + it["bytes"]))
    assert len(got) == k * k
    for iv in got.values():
        iv, ov = _cover(iv)
        assert not ov and _total(iv) == sc * 2


# ---------------------------------------------------------------- all-to-all
def _zipf_counts(k, seed=0):
    rng = np.random.default_rng(seed)
    c = rng.integers(1, 50, size=(k, k)) * (np.arange(k)[None, :] == 0) * 20 + rng.integers(0, 40, size=(k, k))
    return c


@pytest.mark.parametrize("interleave", [True, False])
@pytest.mark.parametrize("stage_sync", [True, False])
def test_alltoall_plan_stages_and_coverage(interleave, stage_sync):
    k = 8
    counts = _zipf_counts(k)
    cfg = hoc.Config(path="ce", chunk_bytes=1024, a2a_interleave=interleave, a2a_stage_sync=stage_sync)
    items = hoc.plan_query(k, hoc.OP_ALLTOALL, 0, hoc.BFLOAT16, counts=counts, config=cfg)
    flows = defaultdict(list)
    per_stage = defaultdict(set)
    for it in items:
        s, d = it["src_rank"], it["dst_rank"]
        assert it["stage"] == (d - s) % k                      # shift stage s holds u -> u+s
        per_stage[it["stage"]].add((s, d))
        flows[(s, d)].append((it["src_off"], it["src_off"] + it["bytes"]))
    for st, pairs in per_stage.items():                         # Eq. 8: one out / one in per rank
        assert len({s for s, _ in pairs}) == len(pairs) == len({d for _, d in pairs})
    for s in range(k):                                          # Eq. 7: the stages cover C exactly
        for d in range(k):
            iv, ov = _cover(flows.get((s, d), []))
            assert not ov and _total(iv) == counts[s][d] * 2
    if stage_sync:
        first = {}
        for it in items:
            first.setdefault(it["step"], it)
        for it in first.values():
            if it["stage"] > 0:
                assert it["n_waits"] >= 1 and first[it["wait0"]]["stage"] < it["stage"]


def test_random_alltoall_plans_cover_every_flow_exactly():
    """Random shapes: k = 1..16, empty rows and columns, odd chunk sizes, both move paths. Every flow's
    bytes leave send[s] at its prefix-sum displacement and land in recv[d] at its own, exactly once."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        k = int(rng.integers(1, 17))
        counts = rng.integers(0, 400, size=(k, k)) * (rng.random((k, k)) < 0.7)
        if trial % 7 == 0:
            counts[int(rng.integers(0, k)), :] = 0          # a rank that sends nothing
        if trial % 11 == 0:
            counts[:, int(rng.integers(0, k))] = 0          # a rank that receives nothing
        dtype, b = [(hoc.BFLOAT16, 2), (hoc.FLOAT32, 4), (hoc.UINT8, 1)][trial % 3]
        chunk = int(rng.choice([256, 1000, 4096, 65536, 0]))
        path = "ce" if trial % 2 else "tma"
        cfg = hoc.Config(path=path, chunk_bytes=chunk, n_copy_streams=int(rng.integers(1, 5)))
        items = hoc.plan_query(k, hoc.OP_ALLTOALL, 0, dtype, counts=counts, config=cfg)
        src, dst = defaultdict(list), defaultdict(list)
        for it in items:
            key = (it["src_rank"], it["dst_rank"])
            assert it["src_buf"] == hoc.BUF_SEND and it["dst_buf"] == hoc.BUF_RECV
            src[key].append((it["src_off"], it["src_off"] + it["bytes"]))
            dst[key].append((it["dst_off"], it["dst_off"] + it["bytes"]))
        for s_ in range(k):
            for d in range(k):
                n = int(counts[s_][d]) * b
                sd = int(counts[s_][:d].sum()) * b                  # prefix sums in rank order
                rd = int(counts[:s_, d].sum()) * b
                if n == 0:
                    assert (s_, d) not in src, (trial, s_, d)
                    continue
                for iv, at in ((src[(s_, d)], sd), (dst[(s_, d)], rd)):
                    merged, ov = _cover(iv)   # no overlap + total n + first and last byte = exact cover
                    assert not ov and _total(merged) == n, (trial, k, s_, d)
                    assert merged[0][0] == at and merged[-1][1] == at + n, (trial, k, s_, d, at, n)


def test_random_block_plans_cover_exactly():
    """Random k, counts and chunks: the reduce-scatter reduces every block once; the all-gather sends
    every rank's block to every rank once; the allreduce reduces every block once and copies it to the
    k - 1 other ranks once (block partition by the closed form, not the oracle's helper)."""
    rng = np.random.default_rng(12)
    for trial in range(40):
        k = int(rng.integers(1, 17))
        n = int(rng.integers(1, 20)) if trial % 5 == 0 else int(rng.integers(1, 50000))  # n < k: empty blocks
        dtype, b = [(hoc.BFLOAT16, 2), (hoc.FLOAT32, 4), (hoc.INT32, 4)][trial % 3]
        chunk = int(rng.choice([256, 1000, 4096, 0]))
        path = "ce" if trial % 2 else "tma"
        cfg = hoc.Config(path=path, chunk_bytes=chunk)
        # reduce-scatter: recvcount n per rank; block r = elements [r*n, (r+1)*n) of every send buffer
        red = defaultdict(list)
        for it in hoc.plan_query(k, hoc.OP_REDUCE_SCATTER, n, dtype, config=cfg):
            assert it["kind"] in (hoc.ITEM_REDUCE, hoc.ITEM_FUSED)
            red[it["dst_rank"]].append((it["src_off"], it["src_off"] + it["bytes"]))
        for r in range(k):
            iv, ov = _cover(red[r])
            assert not ov and _total(iv) == n * b and iv[0][0] == r * n * b, (trial, r)
        # all-gather: send[s] (n elements) lands at recv[d] + s*n for every (s, d)
        got = defaultdict(list)
        for it in hoc.plan_query(k, hoc.OP_ALLGATHER, n, dtype, config=cfg):
            assert it["dst_off"] - it["src_off"] == it["src_rank"] * n * b
            got[(it["src_rank"], it["dst_rank"])].append((it["src_off"], it["src_off"] + it["bytes"]))
        for s_ in range(k):
            for d in range(k):
                iv, ov = _cover(got[(s_, d)])
                assert not ov and _total(iv) == n * b and iv[0][0] == 0, (trial, s_, d)
        # allreduce on the move path: block r = floor(n/k) + [r < n mod k] elements at prefix offsets
        sizes = [n // k + (1 if r < n % k else 0) for r in range(k)]
        offs = [sum(sizes[:r]) for r in range(k)]
        red, mv = defaultdict(list), defaultdict(list)
        for it in hoc.plan_query(k, hoc.OP_ALLREDUCE, n, dtype, config=cfg):
            if it["kind"] == hoc.ITEM_REDUCE:
                red[it["dst_rank"]].append((it["src_off"], it["src_off"] + it["bytes"]))
            else:
                mv[(it["src_rank"], it["dst_rank"])].append((it["src_off"], it["src_off"] + it["bytes"]))
        for r in range(k):
            iv, ov = _cover(red[r])
            if sizes[r] == 0:
                assert not red[r] and not any(mv[(r, d)] for d in range(k))
                continue
            assert not ov and _total(iv) == sizes[r] * b and iv[0][0] == offs[r] * b, (trial, r)
            for d in range(k):
                if d != r:
                    iv, ov = _cover(mv[(r, d)])
                    assert not ov and _total(iv) == sizes[r] * b and iv[0][0] == offs[r] * b, (trial, r, d)


def test_flow_size_aware_interleave_spreads_small_flows():
    k = 2
    counts = np.array([[0, 8 * 512], [2 * 512, 0]])        # flows of 8 and 2 chunks of 1 KiB (bf16)
    def order(interleave):
        items = hoc.plan_query(k, hoc.OP_ALLTOALL, 0, hoc.BFLOAT16, counts=counts,
                               config=hoc.Config(path="ce", chunk_bytes=1024, n_copy_streams=1,
                                                 a2a_interleave=interleave))
        return [it["src_rank"] for it in items]
    fifo = order(False)
    aware = order(True)
    assert fifo == [0] * 8 + [1] * 2
    # weighted interleave: chunk j of a flow of n chunks is due at (j+1)/n.
    # Big flow: 1/8, 2/8, ..., 8/8; small flow: 1/2, 2/2; ties go to flow 0,
    # so the small flow's chunks sit at positions 4 and 9, not 8 and 9.
    pos = [i for i, s in enumerate(aware) if s == 1]
    assert pos == [4, 9]
    assert sorted(aware) == sorted(fifo)


def test_tma_alltoall_is_one_launch_on_caller_stream():
    counts = _zipf_counts(8, 3)
    items = hoc.plan_query(8, hoc.OP_ALLTOALL, 0, hoc.BFLOAT16, counts=counts, config=hoc.Config(path="tma"))
    assert {it["kind"] for it in items} == {hoc.ITEM_TMA}
    assert {it["stream"] for it in items} == {0} and len({it["step"] for it in items}) == 1


def test_sendrecv_plan_chunks():
    # a 32 MiB activation (the PP workload) is one direct copy on the caller's stream
    items = hoc.plan_query(8, hoc.OP_SENDRECV, 16_777_216, hoc.BFLOAT16,
                           config=hoc.Config(path="ce", chunk_bytes=4 << 20, n_copy_streams=4))
    assert len(items) == 1 and items[0]["stream"] == 0 and items[0]["bytes"] == 32 << 20
    # above 64 MiB the message is chunked and striped over the copy queues
    items = hoc.plan_query(8, hoc.OP_SENDRECV, 64 << 20, hoc.BFLOAT16,
                           config=hoc.Config(path="ce", chunk_bytes=4 << 20, n_copy_streams=4))
    assert len(items) == 32 and {it["stream"] for it in items} == {1, 2, 3, 4}
    iv, ov = _cover([(it["src_off"], it["src_off"] + it["bytes"]) for it in items])
    assert not ov and _total(iv) == 128 << 20


# ------------------------------------------------------------ fault injection
@pytest.mark.parametrize("fault", ["drop_chunk", "dup_chunk", "wrong_order"])
def test_host_fault_injection_breaks_the_plan_invariants(fault, monkeypatch):
    k, n = 4, 1 << 16
    cfg = hoc.Config(path="ce", chunk_bytes=1 << 14)
    good = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.FLOAT32, config=cfg)
    monkeypatch.setenv("HOC_FAULT", fault)
    bad = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.FLOAT32, config=cfg)
    if fault == "drop_chunk":
        assert sum(i["bytes"] for i in bad) < sum(i["bytes"] for i in good)
    elif fault == "dup_chunk":
        assert len(bad) == len(good) + 1
    else:
        assert all(i["n_waits"] == 0 for i in bad) and any(i["n_waits"] for i in good)


def test_bad_config_rejected():
    with pytest.raises(hoc.HocError) as e:
        hoc.plan_query(3, hoc.OP_ALLREDUCE, 10, hoc.FLOAT32, config=hoc.Config(ring_order=[0, 1, 1]))
    assert e.value.code == hoc.ERR_INVALID_ARG
    with pytest.raises(hoc.HocError):
        hoc.plan_query(3, hoc.OP_ALLREDUCE, 10, hoc.FLOAT32, config=hoc.Config(n_copy_streams=17))
    with pytest.raises(hoc.HocError) as e:
        hoc.plan_query(3, hoc.OP_ALLREDUCE, 10, hoc.UINT8)
    assert e.value.code == hoc.ERR_UNSUPPORTED


# ------------------------------------------------------------------ sizes
SPAN = 1 << 40  # largest rank buffer span a call may name


@pytest.mark.parametrize("op,count,dtype", [
    (hoc.OP_ALLREDUCE, SPAN // 2 + 1, hoc.BFLOAT16),
    (hoc.OP_SENDRECV, SPAN + 1, hoc.UINT8),
    (hoc.OP_REDUCE_SCATTER, SPAN // (4 * 8) + 1, hoc.FLOAT32),   # the send span is k * recvcount
    (hoc.OP_ALLGATHER, SPAN // (2 * 8) + 1, hoc.BFLOAT16),      # the recv span is k * sendcount
    (hoc.OP_ALLTOALL, SPAN // 8 + 1, hoc.UINT8),                # uniform: k counts per rank
    (hoc.OP_ALLREDUCE, (1 << 64) - 1, hoc.FLOAT32),             # count * 4 wraps size_t
])
def test_oversized_spans_are_rejected_before_any_plan(op, count, dtype):
    with pytest.raises(hoc.HocError) as e:
        hoc.plan_query(8, op, count, dtype)
    assert e.value.code == hoc.ERR_INVALID_ARG and "2^40" in str(e.value)


def test_span_limit_is_inclusive():
    # exactly 2^40 bytes per rank plans (in 4 MiB chunks: 2^18 per rank buffer)
    items = hoc.plan_query(2, hoc.OP_SENDRECV, SPAN, hoc.UINT8)
    assert sum(it["bytes"] for it in items) == SPAN


@pytest.mark.parametrize("counts", [
    lambda k: [[1 << 62 if (a, d) == (0, 1) else 3 for d in range(k)] for a in range(k)],
    # two counts whose sum wraps 2^64 to a small column total
    lambda k: [[1 << 63 if d == 2 and a in (0, 1) else 5 for d in range(k)] for a in range(k)],
    # each count fits, but one receiver's column is over the span
    lambda k: [[SPAN // 4 if d == 0 else 1 for d in range(k)] for a in range(k)],
])
def test_alltoall_counts_that_overflow_are_rejected(counts):
    k = 8
    with pytest.raises(hoc.HocError) as e:
        hoc.plan_query(k, hoc.OP_ALLTOALL, 0, hoc.UINT8, counts=np.array(counts(k), dtype=np.uint64))
    assert e.value.code == hoc.ERR_INVALID_ARG


def test_chunk_count_per_span_is_bounded():
    n = (1 << 33) // 4  # 8 GiB of fp32 per rank
    with pytest.raises(hoc.HocError) as e:
        hoc.plan_query(8, hoc.OP_ALLREDUCE, n, hoc.FLOAT32, config=hoc.Config(path="ce", chunk_bytes=256))
    assert e.value.code == hoc.ERR_INVALID_ARG and "chunk_bytes" in str(e.value)
    # the same size with the default chunk plans
    assert hoc.plan_query(8, hoc.OP_ALLREDUCE, n, hoc.FLOAT32, config=hoc.Config(path="fused"))


def test_copy_queue_count_follows_copy_size_when_left_to_the_scheduler():
    """n_copy_streams = 0: 8 copy queues while every copy of the call is at most 2 MiB, else 4; an explicit
    count is kept whatever the size."""
    def queues(op, count, config, counts=None):
        items = hoc.plan_query(8, op, count, hoc.UINT8, counts=counts, config=config)
        return {it["stream"] for it in items if it["kind"] == hoc.ITEM_COPY}
    auto = hoc.Config(path="ce")
    assert queues(hoc.OP_ALLGATHER, 1 << 20, auto) == set(range(1, 9))        # 1 MiB blocks: 64 small copies
    assert queues(hoc.OP_ALLGATHER, 2 << 20, auto) == set(range(1, 9))        # exactly the threshold
    assert queues(hoc.OP_ALLGATHER, (2 << 20) + 16, auto) == set(range(1, 5))  # past it: one 2 MiB+16 copy each
    assert queues(hoc.OP_ALLGATHER, 32 << 20, auto) == set(range(1, 5))       # 4 MiB chunks
    assert queues(hoc.OP_ALLGATHER, 1 << 20, hoc.Config(path="ce", n_copy_streams=4)) == set(range(1, 5))
    assert queues(hoc.OP_ALLGATHER, 32 << 20, hoc.Config(path="ce", n_copy_streams=6)) == set(range(1, 7))
    small = np.full((8, 8), 1 << 20, dtype=np.uint64)
    assert queues(hoc.OP_ALLTOALL, 0, auto, small) == set(range(1, 9))
    mixed = small.copy()
    mixed[3, 5] = 5 << 20                                                     # one flow of 4 MiB chunks
    assert queues(hoc.OP_ALLTOALL, 0, auto, mixed) == set(range(1, 5))
    # the allreduce's moves: at 8 ranks its chunks are 4 MiB, so 4 queues; at 16 ranks 2 MiB, so 8
    items = hoc.plan_query(8, hoc.OP_ALLREDUCE, 1 << 27, hoc.BFLOAT16, config=auto)
    assert {it["stream"] for it in items if it["kind"] == hoc.ITEM_COPY} == set(range(1, 5))
    items = hoc.plan_query(16, hoc.OP_ALLREDUCE, 1 << 27, hoc.BFLOAT16, config=auto)
    assert {it["stream"] for it in items if it["kind"] == hoc.ITEM_COPY} == set(range(1, 9))


@pytest.mark.parametrize("path,k,chunk_mib", [("ce", 2, 8), ("ce", 4, 4), ("ce", 8, 4), ("ce", 16, 2), ("ce", 12, 2),
                                              ("tma", 2, 16), ("tma", 4, 4), ("tma", 8, 4), ("tma", 16, 4)])
def test_allreduce_chunk_left_to_the_scheduler_follows_the_rank_count(path, k, chunk_mib):
    """chunk_bytes = 0: copy engines take 32 MiB / k within 2-8 MiB, rounded down to a power of two (k = 12:
    2 MiB), and at most 16 MiB over the queues one chunk's copies use (k = 4: 4 MiB on 4 queues); the TMA
    kernel 64 MiB / k^2 within 4-16 MiB; an explicit size is kept; a block smaller than the chunk is one
    chunk."""
    def reduce_steps(count, cfg):
        items = hoc.plan_query(k, hoc.OP_ALLREDUCE, count, hoc.BFLOAT16, config=cfg)
        return len({it["step"] for it in items if it["kind"] == hoc.ITEM_REDUCE})
    def expect(n, chunk):   # chunks cut from each block's first 4 KiB offset (the first one absorbs the head)
        sizes, offs = o_ring.block_partition(n, k)
        return max(max(1, -(-((o + z) * 2 - min((o + z) * 2, -(-o * 2 // 4096) * 4096)) // chunk))
                   for z, o in zip(sizes, offs))
    n = 1 << 27                                                    # 256 MiB of bf16 per rank
    assert reduce_steps(n, hoc.Config(path=path)) == expect(n, chunk_mib << 20)
    assert reduce_steps(n, hoc.Config(path=path, chunk_bytes=1 << 20)) == expect(n, 1 << 20)
    if k in (2, 4, 8, 16):
        assert expect(n, chunk_mib << 20) == (n // k * 2) // (chunk_mib << 20)
    assert reduce_steps(k * 1024, hoc.Config(path=path)) == 1
    if path == "ce" and k == 8:   # 8 explicit queues: 2 MiB chunks keep the 16 MiB in flight
        assert reduce_steps(n, hoc.Config(path=path, n_copy_streams=8)) == (n // k * 2) // (2 << 20)


# ------------------------------------------------------------ random plans
def test_random_large_allreduce_plans_cover_every_block_once():
    """Random rank counts, element counts up to unaligned megabytes (blocks of many chunks, cut on 4 KiB
    offsets), dtypes, move paths and chunk settings: the reduce segments cover each owner's block once
    (the oracle's partition), every other rank receives each block once, and each move waits for the
    reduce of its own chunk."""
    rng = np.random.default_rng(4321)
    dtypes = [(hoc.BFLOAT16, 2), (hoc.FLOAT32, 4), (hoc.INT32, 4)]
    for _ in range(60):
        k = int(rng.integers(2, 17))
        n = int(rng.choice([rng.integers(1 << 16, 1 << 20), rng.integers(1 << 20, 1 << 23)]))
        code, b = dtypes[int(rng.integers(0, 3))]
        path = ["ce", "tma"][int(rng.integers(0, 2))]
        chunk = int(rng.choice([0, 0, 65536 + 16, 1 << 20, 3 << 20]))
        cfg = hoc.Config(path=path, chunk_bytes=chunk)
        items = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, code, config=cfg)
        sizes, offs = o_ring.block_partition(n, k)
        steps = {}
        red, moves = defaultdict(list), defaultdict(list)
        for it in items:
            steps.setdefault(it["step"], it)
            if it["kind"] == hoc.ITEM_REDUCE:
                red[it["dst_rank"]].append((it["src_off"], it["src_off"] + it["bytes"]))
            else:
                moves[(it["src_rank"], it["dst_rank"])].append((it["src_off"], it["src_off"] + it["bytes"]))
                w = steps[it["wait0"]]
                assert w["kind"] == hoc.ITEM_REDUCE and w["stage"] == it["stage"], (k, n, path, chunk)
                assert it["src_off"] == it["dst_off"]
        for r in range(k):
            if sizes[r] == 0:
                assert not red[r]
                continue
            iv, ov = _cover(red[r])
            assert not ov and _total(iv) == sizes[r] * b and iv[0][0] == offs[r] * b, (k, n, path, chunk, r)
            for d in range(k):
                if d != r:
                    iv, ov = _cover(moves[(r, d)])
                    assert not ov and _total(iv) == sizes[r] * b, (k, n, path, chunk, r, d)


def test_random_large_alltoallv_plans_cut_pieces_on_4_kib_destinations():
    """Random counts up to several chunks (zeros, tiny, unaligned): each flow's pieces cover it once,
    contiguously on both sides, and every piece but a flow's first starts on a 4 KiB destination offset."""
    rng = np.random.default_rng(8765)
    for _ in range(60):
        k = int(rng.integers(1, 9))
        counts = rng.integers(0, 5 << 20, size=(k, k)).astype(np.uint64)
        counts[rng.random((k, k)) < 0.2] = 0
        counts[rng.random((k, k)) < 0.2] = rng.integers(1, 100)
        chunk = int(rng.choice([0, 1 << 20, 3 << 20]))
        items = hoc.plan_query(k, hoc.OP_ALLTOALL, 0, hoc.UINT8, counts=counts,
                               config=hoc.Config(path="ce", chunk_bytes=chunk))
        got = defaultdict(list)
        for it in items:
            if it["kind"] == hoc.ITEM_COPY:
                got[(it["src_rank"], it["dst_rank"])].append((it["dst_off"], it["src_off"], it["bytes"]))
        for a in range(k):
            for d in range(k):
                ps = sorted(got[(a, d)])
                assert sum(p[2] for p in ps) == int(counts[a, d]), (k, a, d)
                for (d0, s0, n0), (d1, s1, n1) in zip(ps, ps[1:]):
                    assert d0 + n0 == d1 and s0 + n0 == s1 and d1 % 4096 == 0, (k, a, d)


def test_allreduce_chunk_rule_at_every_rank_count():
    """chunk_bytes = 0 at k = 2..16 (256 MiB bf16 per rank): the copy engines' chunk is a power of two in
    2-8 MiB whose queues hold at most 16 MiB in flight, the TMA kernel's 4-16 MiB; every chunk after a
    block's first is one whole chunk of that size (the last may be shorter)."""
    n = 1 << 27
    for k in range(2, 17):
        sizes, offs = o_ring.block_partition(n, k)
        for path, lo, hi in (("ce", 2 << 20, 8 << 20), ("tma", 4 << 20, 16 << 20)):
            items = hoc.plan_query(k, hoc.OP_ALLREDUCE, n, hoc.BFLOAT16, config=hoc.Config(path=path))
            segs = defaultdict(list)
            for it in items:
                if it["kind"] == hoc.ITEM_REDUCE:
                    segs[it["dst_rank"]].append((it["src_off"], it["bytes"]))
            chunk = max(nb for r in segs for _, nb in sorted(segs[r])[1:-1]) if len(segs[0]) > 2 else None
            assert chunk is not None and lo <= chunk <= hi, (k, path, chunk)
            if path == "ce":
                assert chunk & (chunk - 1) == 0, (k, chunk)
                queues = {it["stream"] for it in items if it["kind"] == hoc.ITEM_COPY}
                assert chunk * min(len(queues), k * (k - 1)) <= 16 << 20, (k, chunk, len(queues))
            for r in range(k):
                mid = sorted(segs[r])[1:-1]
                assert all(nb == chunk for _, nb in mid), (k, path, r)
