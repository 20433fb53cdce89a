#!/usr/bin/env python
"""Benchmark of the simulated-rank ring allreduce on one GB300.

Workload: ring allreduce (sum) over 8 simulated ranks, 134,217,728 bf16
elements (256 MiB) per rank drawn N(0, 1e-3), fp32 accumulation, every rank
buffer resident in one GPU's HBM.  One step = one allreduce through the C ABI
(plan lookup, stream fork/join, k-way reduce, all-gather moves).

Prints one JSON line: bus bandwidth (nccl-tests convention, 2(k-1)/k * S / t)
as `value`, plus the HBM-roofline fraction of the executed schedule, SMs
used, the probe-kernel slowdown per path, the end-to-end figure through host
buffers, the clocks seen during the timed region, and the CPU oracle timed on
a sample of the same workload.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path does not shard): `value` = all ranks' bus bytes / max time.

`--impl reference` times the CPU oracle (the slow reference implementation)
on a bounded sample instead; only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

# The host proxy's copies must not share a hardware work queue with a stream
# held at its start flag (see include/hoc_proxy.h); set before CUDA starts.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "simulated-rank allreduce bus GB/s & % HBM roofline; SMs used; probe slowdown"
K_RANKS = 8
N_ELEMS = 134_217_728
SIGMA = 1e-3
WORKLOAD = ("ring allreduce (sum), 8 simulated ranks, 134,217,728 bf16 elements (256 MiB) per rank, "
            "N(0, 1e-3), fp32 accumulation")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, nominal


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="auto", choices=["auto", "ce", "tma", "fused"])
    ap.add_argument("--chunk-bytes", type=int, default=0, help="0: picked by the scheduler (allreduce: by move path and rank count)")
    ap.add_argument("--copy-streams", type=int, default=0, help="0: picked per call by copy size (8 or 4 queues)")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-path, probe and e2e legs")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--mode", default="allreduce", choices=["allreduce", "allgather", "ep_fused"],
                    help="allgather: time only the all-gather moves of the workload's 32 MiB blocks "
                         "(a profiling case: the copy-engine path launches no kernel); ep_fused: time only the "
                         "EP dispatch + combine fused with the exchange (8 ranks x 4096 tokens x 2048, top-6 of 64)")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="skip the DP bucket stream, 1F1B pipeline and EP dispatch/combine legs")
    ap.add_argument("--count", type=int, default=N_ELEMS,
                    help="elements per rank (default: the full 134,217,728; smaller only for profiling captures)")
    return ap.parse_args()


# --------------------------------------------------------------------- inputs
def _gen_rank(args):
    from collective_communication_schedules_gb300 import inputs
    r, n = args
    return inputs.normal_bf16(n, inputs.seed_for(2, 0, r), SIGMA)


def generate_inputs(k: int, n: int):
    """Seeded inputs, one process per rank (spawned before any CUDA call)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor

    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))  # replicas on this host share its cores
    workers = max(1, min(k, (os.cpu_count() or 1) // max(1, local_ranks)))
    with ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(_gen_rank, [(r, n) for r in range(k)]))


# --------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(dev: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[dev] if dev < len(ids) else str(dev)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel: str, k: int, count: int):
    """DRAM bytes per launch from a committed ncu summary, if it matches today's kernel source and workload."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e or e.get("k") != k or e.get("count") != count:
        return None
    src = os.path.join(ROOT, "collective_communication_schedules_gb300", "csrc", e.get("source", "reduce.cu"))
    try:
        digest = hashlib.sha256(source_code(open(src).read())).hexdigest()[:16]
    except OSError:
        return None
    return e.get("bytes_per_launch") if digest == e.get("code_sha256_16") else None


def source_code(text: str) -> bytes:
    """A source file's code without its // comments and blank lines: what the counters depend on."""
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln).encode()


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = os.environ.get("HOC_DIST_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bus_bytes(k: int, per_rank_bytes: int) -> float:
    return 2.0 * (k - 1) / k * per_rank_bytes


# ------------------------------------------------------------- CPU baseline
CPU_SAMPLE = 8 << 20   # elements per rank the oracle folds: the first 8,388,608 of every rank's buffer


def cpu_sample_text(reps=None, secs=None):
    """The one definition of the oracle's sample, shared by cpu_baseline and the reference arm."""
    s = (f"numpy ring-order fold of the first {CPU_SAMPLE:,} of the {N_ELEMS:,} bf16 elements per rank "
         f"(8 ranks, 1/{N_ELEMS // CPU_SAMPLE} of the workload)")
    if reps is not None:
        s += f", {reps} repetitions, {secs:.3f} s each"
    return s + f"; host has {os.cpu_count()} cores, numpy elementwise runs on 1"


def oracle_config():
    """`config` of both arms: the workload, not how either arm runs it."""
    return {"workload": WORKLOAD, "k": K_RANKS, "count": N_ELEMS,
            "l2": "no flush: each step reads 2 GiB of inputs and writes 2 GiB, > 129 MB L2",
            "parallelism": "independent replicas, one per GPU"}


def cpu_baseline(xs_host, seconds: float, device_out=None):
    """The oracle, as it stands, on the CPU_SAMPLE elements at the start of every rank's buffer."""
    import numpy as np

    from oracle import ring

    n = CPU_SAMPLE
    xs = [x[:n] for x in xs_host]
    t0 = time.perf_counter()
    reps = 0
    y = None
    while True:
        y = ring.allreduce(xs, "bfloat16")
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / reps
    out = {"value": round(bus_bytes(K_RANKS, n * 2) / dt / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": cpu_sample_text(reps, dt), "seconds_per_step": round(dt, 4)}
    if device_out is not None:
        # The GPU result on the same sample must equal the oracle bit for bit.
        import torch
        rng = np.random.default_rng(123)
        idx = np.sort(rng.choice(n, size=min(n, 1 << 20), replace=False))
        try:
            ti = torch.from_numpy(idx).to(device_out[0].device)
            ok = True
            for r in range(K_RANKS):
                got = device_out[r].view(torch.int16).index_select(0, ti).cpu().numpy().view(np.uint16)
                ok = ok and bool(np.array_equal(got, y[r][idx]))
            out["parity_sample_ok"] = ok
        except Exception as e:  # noqa: BLE001 -- reported; the baseline's timing stands
            out["parity_sample_ok"] = None
            out["parity_error"] = f"{type(e).__name__}: {e}"
    return out


def cpu_baseline_buckets(host_pool, buckets: int = 16):
    """The oracle's reduce-scatter on the first `buckets` of the DP stream's 16 pool buckets, timed on
    the host, and the per-bucket time scaled to the stream's 268 buckets (labelled as scaled)."""
    from oracle import ring

    k, be = K_RANKS, 13_107_200
    t0 = time.perf_counter()
    for s in range(buckets):
        ring.reduce_scatter([host_pool[s * k + r] for r in range(k)], be // k, "bfloat16")
    per = (time.perf_counter() - t0) / buckets
    return {"kind": "oracle", "cores": 1, "ms_per_bucket": round(per * 1e3, 2),
            "ms_total_scaled": round(per * 268 * 1e3, 1),
            "rs_bus_gbs": round((k - 1) / k * be * 2 / per / 1e9, 3),
            "sample": f"{buckets} of the 16 pool buckets (8 ranks x 13,107,200 bf16 each), timed, total scaled "
                      f"x268/{buckets}"}


def run_reference(args, world, rank):
    """--impl reference: the oracle as the reference arm (rank 0 only), on the same sample as cpu_baseline."""
    if rank != 0:
        return
    from collective_communication_schedules_gb300 import inputs
    from oracle import ring

    n = CPU_SAMPLE
    xs = [inputs.normal_bf16(n, inputs.seed_for(2, 0, r), SIGMA) for r in range(K_RANKS)]   # the draws' first n
    for _ in range(args.warmup):
        ring.allreduce(xs, "bfloat16")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ring.allreduce(xs, "bfloat16")
    dt = (time.perf_counter() - t0) / args.steps
    v = bus_bytes(K_RANKS, n * 2) / dt / 1e9
    line = {"metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": oracle_config(), "impl": "reference",
            "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": cpu_sample_text() + "; one fold per step"},
            "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU legs
def time_allreduce(comm, send, recv, stream, steps, profile_kind=None):
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        comm.allreduce(send, recv, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


PROBE_SHAPES = {
    # small CTAs (8 x 256 threads per SM per wave) that can share an SM with a collective's CTAs
    "coresident": dict(ctas_per_sm=8, threads=256, whole_sm=False),
    # CTAs that hold a whole SM (all registers, nearly all shared memory), as a GEMM tile does
    "whole_sm": dict(ctas_per_sm=1, threads=1024, whole_sm=True),
}
PROBE_KERNELS = 40          # the probe is a train of one-wave kernels, ~0.25 ms each


def probe_slowdown(run_coll, coll_ms: float, stream_c, sms: int, shape: str = "whole_sm", n_kernels: int = 0,
                   priority: int = 0, graph: bool = False, pdl: bool = False):
    """Slowdown of the FMA probe train while the collective runs back to back beside it.

    The probe is a train of short one-wave kernels, like a sequence of layer
    kernels: between two probe kernels the block scheduler hands SMs to
    whichever kernel launched first, so a collective that needs SMs takes them
    from the probe, and one that needs none (copy engines) leaves it alone.
    `priority`: the probe stream's priority (lower is higher, as for CUDA);
    `graph`: the train is captured once into a CUDA graph and replayed;
    `pdl`: each probe kernel is launched with programmatic dependent launch
    (it waits for the one before it, only the launch overlaps).
    """
    import torch

    from collective_communication_schedules_gb300 import hoc

    cfg = PROBE_SHAPES[shape]
    ctas, threads, whole = cfg["ctas_per_sm"] * sms, cfg["threads"], cfg["whole_sm"]
    nk = n_kernels or PROBE_KERNELS
    sp = torch.cuda.Stream(priority=priority)
    gate = torch.cuda.Stream()
    sink = torch.zeros(4, dtype=torch.float32, device="cuda")
    mhz = []
    trains = {}

    def capture(iters):   # the train as one CUDA graph, captured before the timed runs
        if graph and iters not in trains:
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=sp):
                for _ in range(nk):
                    hoc.probe_launch(ctas, threads, iters, stream=sp, whole_sm=whole, sink=sink, pdl=pdl)
            trains[iters] = g
            torch.cuda.synchronize()

    def train(iters):
        if graph:
            with torch.cuda.stream(sp):
                trains[iters].replay()
        else:
            for _ in range(nk):
                hoc.probe_launch(ctas, threads, iters, stream=sp, whole_sm=whole, sink=sink, pdl=pdl)

    def run_probe(iters, with_coll=False, n_coll=0):
        capture(iters)
        ev_gate = torch.cuda.Event()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        hoc.probe_launch(sms, 256, 60000, stream=gate)      # ~1 ms gate: both streams start together
        ev_gate.record(gate)
        sp.wait_event(ev_gate)
        stream_c.wait_event(ev_gate)
        if with_coll:
            for _ in range(n_coll):
                run_coll(stream_c)
        a.record(sp)
        train(iters)
        b.record(sp)
        torch.cuda.synchronize()
        cyc, ns = sink[0].item(), sink[1].item()
        mhz.append(1e3 * cyc / ns if ns > 0 else None)
        return a.elapsed_time(b)

    base = run_probe(100)
    iters = max(100, int(100 * 10.0 / max(base, 1e-3)))      # ~10 ms for the whole train alone
    mhz.clear()
    alone = statistics.median(run_probe(iters) for _ in range(3))
    mhz_alone = [m for m in mhz if m]
    mhz.clear()
    n_coll = int(math.ceil(1.5 * alone / max(coll_ms, 1e-3))) + 2
    with_c = statistics.median(run_probe(iters, True, n_coll) for _ in range(3))
    mhz_with = [m for m in mhz if m]
    return {"shape": f"{nk} kernels x {ctas} CTAs x {threads} threads" + (", whole SM each" if whole else "")
                     + (", programmatic dependent launches" if pdl else ""),
            "probe_alone_ms": round(alone, 3), "probe_with_ms": round(with_c, 3),
            "slowdown": round(with_c / alone - 1.0, 4), "collectives_beside": n_coll,
            "sm_mhz_alone": round(statistics.median(mhz_alone), 1) if mhz_alone else None,
            "sm_mhz_with": round(statistics.median(mhz_with), 1) if mhz_with else None}


def probes(run_coll, coll_ms, stream_c, sms, n_kernels=0, priority=0, graph=False, pdl=False):
    return {shape: probe_slowdown(run_coll, coll_ms, stream_c, sms, shape, n_kernels, priority, graph, pdl)
            for shape in PROBE_SHAPES}


def leg_ce_interference(send, recv, n_el, k, local, stream, sms):
    """What slows the probe train beside copy-engine moves that use no SM.

    (a) the same probe work as 10 / 40 / 160 kernels beside the default moves:
        a cost paid per kernel launch grows with the count;
    (b) copy size x copy queues of the all-gather moves (8 x 32 MiB blocks);
    (c) the probe's own SM clock (cycles / ns in its first CTA) with each;
    (d) 512 KiB copies whose buffers stay in L2 against 512 KiB copies through HBM:
        separates the copies' HBM traffic from their number and size;
    (e) the default moves issued copy by copy instead of as one CUDA graph per call.
    """
    import torch

    from collective_communication_schedules_gb300 import hoc

    blk = n_el // k

    def moves(chunk, nq, block=blk, graphs=True):
        c = hoc.Comm(k, local, hoc.Config(path="ce", chunk_bytes=chunk, n_copy_streams=nq, use_graphs=graphs))
        s_ = [t[:block] for t in send]
        r_ = [t[:k * block] for t in recv]
        run = lambda st, c=c: c.allgather(s_, r_, stream=st)
        for _ in range(3):
            run(stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            run(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 10
        st = c.last_stats()
        return c, run, ms, {"ms": round(ms, 4), "bytes_gbs": round(st["bytes_exec"] / (ms * 1e-3) / 1e9, 1),
                            "copies_per_call": st["copies"], "kernels_per_call": st["kernels"]}

    def slow(pr):
        return {sh: pr[sh]["slowdown"] for sh in pr}

    def mhz(pr):
        return {sh: [pr[sh]["sm_mhz_alone"], pr[sh]["sm_mhz_with"]] for sh in pr}

    out = {"launch_count": [], "copy_shape": [], "l2_vs_hbm": [], "issue": []}
    c, run, ms, info = moves(4 << 20, 4)
    for nk in (10, 40, 160):
        pr = probes(run, ms, stream, sms, nk)
        out["launch_count"].append({"probe_kernels": nk, "slowdown": slow(pr), "sm_mhz_alone_with": mhz(pr),
                                    "probe_alone_ms": {sh: pr[sh]["probe_alone_ms"] for sh in pr}})
    c.close()
    for mib, nq in ((4, 4), (4, 2), (4, 3), (2, 4), (2, 8), (8, 2), (8, 1), (16, 1), (4, 8), (8, 8), (16, 16)):
        c, run, ms, info = moves(mib << 20, nq)
        pr = probes(run, ms, stream, sms)
        out["copy_shape"].append(dict(chunk_mib=mib, copy_streams=nq, slowdown=slow(pr), sm_mhz_alone_with=mhz(pr),
                                      **info))
        c.close()
    small = 512 << 10
    for label, block in (("l2_resident", small), ("hbm", blk)):
        # l2_resident: 8 blocks of 512 KiB gathered to 8 ranks (36 MiB in all, inside L2)
        c, run, ms, info = moves(small, 4, block=block)
        pr = probes(run, ms, stream, sms)
        out["l2_vs_hbm"].append(dict(buffers=label, chunk_kib=512, copy_streams=4, slowdown=slow(pr), **info))
        c.close()
    for graphs in (True, False):
        c, run, ms, info = moves(4 << 20, 4, graphs=graphs)
        pr = probes(run, ms, stream, sms)
        out["issue"].append(dict(graphs=graphs, slowdown=slow(pr), **info))
        c.close()
    # (f) the probe's stream at the highest priority; (g) the probe train launched as one CUDA graph
    out["probe_side"] = []
    c, run, ms, info = moves(4 << 20, 4)
    for label, kw in (("high_priority_stream", dict(priority=-100)), ("graph_launched_train", dict(graph=True)),
                      ("both", dict(priority=-100, graph=True))):
        pr = probes(run, ms, stream, sms, **kw)
        out["probe_side"].append(dict(probe=label, slowdown=slow(pr), sm_mhz_alone_with=mhz(pr), **info))
    c.close()
    return out


# ------------------------------------------------------ the other workloads
def _gen_bucket(args):
    from collective_communication_schedules_gb300 import inputs
    slot, r = args
    return inputs.normal_bf16(13_107_200, inputs.seed_for(3, slot, r), SIGMA)


def leg_bucket_stream(host_pool, sms, peak):
    """8 ranks, 268 reduce-scatters of 25 MiB buckets back to back, probe beside; SM budget sweep."""
    import torch

    from collective_communication_schedules_gb300 import hoc

    k, nb, be, pool = 8, 268, 13_107_200, 16
    rc = be // k
    dev = torch.device("cuda")
    pool_in = [[torch.from_numpy(host_pool[s * k + r].view("int16")).view(torch.bfloat16).to(dev)
                for r in range(k)] for s in range(pool)]
    outs = torch.empty((nb, k, rc), dtype=torch.bfloat16, device=dev)
    # each bucket's k output views, made once: building them per call costs more host time than the call
    out_views = [[outs[b, r] for r in range(k)] for b in range(nb)]
    stream = torch.cuda.Stream()
    out = {"buckets": nb, "bucket_bytes_per_rank": be * 2, "budgets": []}
    for m, eng in ((4, "lsu"), (4, "tma"), (8, "lsu"), (8, "tma"), (16, "lsu"), (16, "tma"), (32, "lsu"),
                   (32, "tma"), (0, "lsu"), (0, "tma")):
        with hoc.Comm(k, torch.cuda.current_device(), hoc.Config(reduce_max_sms=m, reduce_engine=eng)) as c:
            def run(s, c=c):
                for b in range(nb):
                    c.reduce_scatter(pool_in[b % pool], out_views[b], rc, stream=s)
            run(stream)
            torch.cuda.synchronize()
            runs = []
            for _ in range(3):  # the median of three streams of 268 buckets
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run(stream)
                e1.record(stream)
                torch.cuda.synchronize()
                runs.append(e0.elapsed_time(e1))
            ms = statistics.median(runs)
            st = c.last_stats()
            per = ms / nb
            entry = {"reduce_max_sms": m or sms, "engine": eng, "ms_total": round(ms, 3), "ms_per_bucket": round(per, 4),
                     "rs_bus_gbs": round((k - 1) / k * be * 2 / (per * 1e-3) / 1e9, 1),
                     "hbm_frac": round(st["bytes_exec"] / (per * 1e-3) / (peak * 1e9), 4),
                     "sms_used": st["sms_used"]}
            entry["probe"] = probes(run, ms, stream, sms)
            out["budgets"].append(entry)
    # the whole stream of 268 reduce-scatters (whole GPU) captured once into a CUDA graph and replayed:
    # one launch for the stream instead of 268 host calls
    try:
        out["graph_replay"] = _bucket_stream_graph(hoc, torch, k, nb, pool, rc, pool_in, out_views, stream, peak)
    except Exception as e:  # reported in the line; the other legs stand
        torch.cuda.synchronize()
        out["graph_replay"] = {"error": str(e)}
    del pool_in, outs, out_views
    torch.cuda.empty_cache()
    return out


def _bucket_stream_graph(hoc, torch, k, nb, pool, rc, pool_in, out_views, stream, peak):
    with hoc.Comm(k, torch.cuda.current_device()) as c:
        def run_all(s, c=c):
            for b in range(nb):
                c.reduce_scatter(pool_in[b % pool], out_views[b], rc, stream=s)
        run_all(stream)                                    # plans built before the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            run_all(stream)
        runs = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):  # replay() launches on the current stream
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            runs.append(e0.elapsed_time(e1))
        ms = statistics.median(runs)
        res = {"ms_total": round(ms, 3), "ms_per_bucket": round(ms / nb, 4),
               "hbm_frac": round(c.last_stats()["bytes_exec"] / (ms / nb * 1e-3) / (peak * 1e9), 4)}
        del graph
    return res


def leg_pipeline(sms):
    """8 stages x 16 micro-batches of 32 MiB bf16 activations in 1F1B order."""
    import torch

    from collective_communication_schedules_gb300 import hoc, inputs
    from collective_communication_schedules_gb300.pipeline import Pipeline1F1B

    p, m, elems = 8, 16, 4096 * 4096
    keys = inputs.pp_keys(p, m)
    g = torch.Generator(device="cuda").manual_seed(4100)
    xs = [torch.randn(elems, generator=g, device="cuda").to(torch.bfloat16) for _ in range(m)]
    out = {}
    first = None  # results of the first run with sends: every mode and path must give the same bits
    same = True
    for path in ("ce", "tma"):
        with hoc.Comm(p, torch.cuda.current_device(), hoc.Config(path=path)) as c:
            res = {}
            # sends completed by events (the sender keeps computing), sends on the sender's stream, no sends
            for label, mode in (("pull_sends", "pull"), ("event_sends", "event"), ("stream_sends", "stream"),
                                ("compute_only", None)):
                pipe = Pipeline1F1B(c, p, m, elems, keys, probe_ctas=2 * sms, probe_iters=2000, sends=mode or "stream")
                if mode is None:
                    pipe.comm = _NoSend()
                runs = []
                for _ in range(3):
                    pipe.load(xs)
                    torch.cuda.synchronize()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    pipe.issue()
                    e1.record()
                    torch.cuda.synchronize()
                    runs.append(e0.elapsed_time(e1))
                res[label + "_ms"] = round(statistics.median(runs), 3)
                if mode is not None:
                    if first is None:
                        first = [pipe.result(i).clone() for i in range(m)]
                    else:
                        same = same and all(torch.equal(pipe.result(i).view(torch.int16), first[i].view(torch.int16))
                                            for i in range(m))
                del pipe
                torch.cuda.empty_cache()
            sends = 2 * (p - 1) * m
            res["sends"] = sends
            res["send_bytes"] = sends * elems * 2
            res["exposed_ms_pull_sends"] = round(res["pull_sends_ms"] - res["compute_only_ms"], 3)
            res["exposed_ms_event_sends"] = round(res["event_sends_ms"] - res["compute_only_ms"], 3)
            res["exposed_ms_stream_sends"] = round(res["stream_sends_ms"] - res["compute_only_ms"], 3)
            out[path] = res
    out["results_identical_across_modes_and_paths"] = bool(same)
    return out


class _NoSend:
    """Stands in for the communicator to time the pipeline's compute alone."""

    def sendrecv(self, *a, **kw):
        return None

    def sendrecv_async(self, *a, stream=None, done=None, **kw):
        done.record(stream)
        return done


def leg_expert_dispatch(peak):
    """8 ranks x 4096 tokens x 2048 bf16, top-6 of 64 experts (Zipf 1.1): dispatch + combine."""
    import numpy as np
    import torch

    from collective_communication_schedules_gb300 import hoc, inputs

    w = inputs.EP_DISPATCH
    k, h = w["k"], w["hidden"]
    routing = inputs.ep_routing(k, w["tokens"], w["experts"], w["topk"], w["zipf"])
    counts = np.zeros((k, k), dtype=np.int64)
    for r in range(k):
        counts[r] = np.bincount(routing[r].reshape(-1) // (w["experts"] // k), minlength=k)
    ecounts = counts * h
    rows = counts.sum(axis=1)
    g = torch.Generator(device="cuda").manual_seed(5500)
    send = [torch.randn(int(rows[r]) * h, generator=g, device="cuda").to(torch.bfloat16) for r in range(k)]
    recv = [torch.empty(int(ecounts[:, d].sum()), dtype=torch.bfloat16, device="cuda") for d in range(k)]
    back = [torch.empty_like(t) for t in send]
    moved = int(ecounts.sum()) * 2
    out = {"rows_per_dst": [int(v) for v in counts.sum(axis=0)], "bytes_per_direction": moved}
    for path, inter in (("ce", True), ("ce", False), ("tma", True)):
        with hoc.Comm(k, torch.cuda.current_device(), hoc.Config(path=path, a2a_interleave=inter)) as c:
            def run(c=c):
                c.alltoall(send, recv, sendcounts=ecounts, dtype=hoc.BFLOAT16)
                c.alltoall(recv, back, sendcounts=ecounts.T.copy(), dtype=hoc.BFLOAT16)
            run()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                run()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / 5
            st = c.last_stats()
            # tail of the dispatch: when each copy stream finished, from the fork
            c.profile_enable(True)
            c.alltoall(send, recv, sendcounts=ecounts, dtype=hoc.BFLOAT16)
            fin = c.profile_stream_finish()
            c.profile_enable(False)
            torch.cuda.synchronize()
            tail = {}
            if fin:
                tail = {"stream_finish_ms": [round(v, 4) for v in fin],
                        "finish_spread_ms": round(max(fin) - min(fin), 4),
                        "last_over_mean": round(max(fin) / (sum(fin) / len(fin)), 3)}
            out[f"{path}{'' if inter else '_fifo'}"] = {
                "dispatch_plus_combine_ms": round(ms, 4),
                "algbw_gbs": round(2 * moved / (ms * 1e-3) / 1e9, 1),
                "hbm_frac": round(2 * st["bytes_exec"] / (ms * 1e-3) / (peak * 1e9), 4),
                "sms_used": st["sms_used"], "copies_per_call": st["copies"], "dispatch_tail": tail}
    ok = all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(send, back))
    out["combine_restores_dispatch_input"] = bool(ok)

    # The whole round on the device, with no host synchronisation: pack kernels,
    # dispatch with device-computed counts (stream-memop handshake with the host
    # proxy), the inverse exchange, and the weighted top-k combine kernel.
    tokens, topk, experts = w["tokens"], w["topk"], w["experts"]
    s = torch.cuda.Stream()
    xs = [torch.randn((tokens, h), generator=g, device="cuda").to(torch.bfloat16) for _ in range(k)]
    ids = [torch.from_numpy(routing[r].astype(np.int32)).cuda() for r in range(k)]
    gate = [torch.rand(tokens * topk, generator=g, device="cuda") for _ in range(k)]
    n = tokens * topk
    psend = [torch.empty((n, h), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    perm = [torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(k)]
    pos = [torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(k)]
    wsp = [torch.empty(hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda") for _ in range(k)]
    d_counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    cap = [int(ecounts[:, d].sum()) for d in range(k)]
    precv = [torch.empty(cap[d], dtype=torch.bfloat16, device="cuda") for d in range(k)]
    pback = [torch.empty(n * h, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    ys = [torch.empty((tokens, h), dtype=torch.bfloat16, device="cuda") for _ in range(k)]

    ids_flat = [t.view(-1) for t in ids]
    wsp_all = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    st_all = torch.zeros(1, dtype=torch.int32, device="cuda")

    def pack_all():    # every rank's pack in one set of launches
        hoc.ep_pack_all(ids_flat, xs, experts, [t.view(-1) for t in psend], [n * h] * k, pos, d_counts, wsp_all,
                        st_all, stream=s)

    def combine_all():
        hoc.ep_combine_all(pback, [n * h] * k, pos, gate, tokens, topk, h, ys, st_all, stream=s)

    def device_round_trip():
        with hoc.Comm(k, torch.cuda.current_device()) as c:
            def round_trip():
                pack_all()
                c.alltoall_device_counts([t.view(-1) for t in psend], precv, d_counts, cap, hoc.BFLOAT16, stream=s)
                c.alltoall_device_counts(precv, pback, d_counts, [n * h] * k, hoc.BFLOAT16, stream=s, transpose=True)
                combine_all()
            round_trip()
            c.wait(s, timeout_ms=60000)
            host_us = []
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            for _ in range(5):
                t0 = time.perf_counter()
                round_trip()
                host_us.append((time.perf_counter() - t0) * 1e6)
            e1.record(s)
            c.wait(s, timeout_ms=60000)
            ms = e0.elapsed_time(e1) / 5
            # one more round with an event between its phases (all on stream s), queued
            # behind a spin kernel so that the host's issue time stays out of the phases
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            gpu_spin(s, 2.0)
            ev[0].record(s)
            pack_all()
            ev[1].record(s)
            c.alltoall_device_counts([t.view(-1) for t in psend], precv, d_counts, cap, hoc.BFLOAT16, stream=s)
            ev[2].record(s)
            c.alltoall_device_counts(precv, pback, d_counts, [n * h] * k, hoc.BFLOAT16, stream=s, transpose=True)
            ev[3].record(s)
            combine_all()
            ev[4].record(s)
            # the same pack and combine rank by rank (one set of launches per rank), for comparison
            ev2 = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            gpu_spin(s, 2.0)
            ev2[0].record(s)
            for r in range(k):
                hoc.ep_pack(ids[r], xs[r], experts, k, psend[r], perm[r], pos[r], d_counts[r], wsp[r], stream=s)
            ev2[1].record(s)
            c.alltoall_device_counts([t.view(-1) for t in psend], precv, d_counts, cap, hoc.BFLOAT16, stream=s)
            c.alltoall_device_counts(precv, pback, d_counts, [n * h] * k, hoc.BFLOAT16, stream=s, transpose=True)
            ev2[2].record(s)
            for r in range(k):
                hoc.ep_combine(pback[r], pos[r], gate[r], tokens, topk, h, ys[r], stream=s)
            ev2[3].record(s)
            c.wait(s, timeout_ms=60000)
            phases = {name: round(ev[i].elapsed_time(ev[i + 1]), 4) for i, name in
                      enumerate(("pack_ms", "dispatch_ms", "combine_exchange_ms", "combine_kernel_ms"))}
            per_rank = {"pack_ms": round(ev2[0].elapsed_time(ev2[1]), 4),
                        "combine_kernel_ms": round(ev2[2].elapsed_time(ev2[3]), 4)}
            st = c.proxy_status()
        return {
            "ms": round(ms, 4), "host_issue_us": round(statistics.median(host_us), 1), "phases": phases,
            "pack_and_combine_rank_by_rank": per_rank, "status": int(st_all.item()),
            "steps": "pack of every rank (one set of launches) -> dispatch (device counts, host proxy, copy engines) "
                     "-> combine exchange (copy engines) -> weighted combine of every rank",
            "proxy_tasks_completed": st["completed"], "proxy_tasks_released_on_error": st["released_on_error"]}

    try:
        out["device_round_trip"] = device_round_trip()
    except hoc.HocError as e:  # reported in the line; the other legs stand
        torch.cuda.synchronize()
        out["device_round_trip"] = {"error": str(e)}

    # The same round trip fused with the exchange: the dispatch scatters every
    # token row straight into the destination ranks' receive buffers and the
    # combine reads the rows where the experts left them (SMs; no send buffer,
    # no copies).  Identity experts, as above; the results must be the same bits.
    fcap = [int(ecounts[:, d].sum()) for d in range(k)]
    frecv = [torch.empty(fcap[d], dtype=torch.bfloat16, device="cuda") for d in range(k)]
    fpos = [torch.empty(n, dtype=torch.int32, device="cuda") for _ in range(k)]
    fcounts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    fws = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    fstatus = torch.zeros(1, dtype=torch.int32, device="cuda")
    fys = [torch.empty((tokens, h), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    ids_flat = [t.view(-1) for t in ids]

    def fused_once():
        hoc.ep_dispatch_fused(ids_flat, xs, experts, frecv, fcap, fpos, fcounts, fws, fstatus, stream=s)
        hoc.ep_combine_fused(frecv, fcap, ids_flat, fpos, fcounts, gate, tokens, topk, h, experts, fys, fstatus,
                             stream=s)

    fused_once()
    torch.cuda.synchronize()
    host_us = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(10):
        t0 = time.perf_counter()
        fused_once()
        host_us.append((time.perf_counter() - t0) * 1e6)
    e1.record(s)
    torch.cuda.synchronize()
    f_ms = e0.elapsed_time(e1) / 10
    ph = []
    for _ in range(5):  # phases: dispatch (sort + scatter), combine; queued behind a spin kernel
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        gpu_spin(s, 1.0)
        ev[0].record(s)
        hoc.ep_dispatch_fused(ids_flat, xs, experts, frecv, fcap, fpos, fcounts, fws, fstatus, stream=s)
        ev[1].record(s)
        hoc.ep_combine_fused(frecv, fcap, ids_flat, fpos, fcounts, gate, tokens, topk, h, experts, fys, fstatus,
                             stream=s)
        ev[2].record(s)
        torch.cuda.synchronize()
        ph.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
    d_ms = statistics.median(p[0] for p in ph)
    c_ms = statistics.median(p[1] for p in ph)
    rows_moved = int(ecounts.sum()) // h                     # valid (token, slot) pairs of all ranks
    row_b = h * 2
    disp_bytes = k * tokens * row_b + rows_moved * row_b + k * n * 12      # rows read once, written per pair; ids, pos
    comb_bytes = rows_moved * row_b + k * tokens * row_b + k * n * 12      # rows read per pair, outputs written; ids, pos, w
    same = all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(fys, ys))
    out["fused_round_trip"] = {
        "ms": round(f_ms, 4), "host_issue_us": round(statistics.median(host_us), 1),
        "phases": {"dispatch_ms": round(d_ms, 4), "combine_ms": round(c_ms, 4)},
        "dispatch_bytes": disp_bytes, "combine_bytes": comb_bytes,
        "dispatch_hbm_frac": round(disp_bytes / (d_ms * 1e-3) / (peak * 1e9), 4),
        "combine_hbm_frac": round(comb_bytes / (c_ms * 1e-3) / (peak * 1e9), 4),
        "phase_timing": "events between the phases, the launches queued behind a spin kernel (host issue time "
                        "excluded); the dispatch phase includes the sort",
        "status": int(fstatus.item()), "results_equal_copy_engine_round_trip": bool(same),
        "steps": "fused dispatch (sort of every rank's pairs, rows scattered into the receive buffers) -> "
                 "fused combine (rows read in place from the expert ranks' buffers)",
        "kernels": 5, "copies": 0}
    return out


SWEEP_ROTATION_BYTES = 320 << 20   # > 2x the 126 MB L2: each timed pass cycles through this much memory


def _sweep_call(c, hoc, op, src, dst, k, n, reg, stream):
    """One op of the sweep on region `reg` of the rank buffers (every region is n bytes per rank)."""
    o = reg * n
    if op == "p2p":
        c.sendrecv(0, src[0][o:], 1, dst[1][o:], n, hoc.UINT8, stream=stream)
    elif op == "allgather":
        cs = n // k
        c.allgather([t[reg * cs:] for t in src], [t[o:] for t in dst], cs, hoc.UINT8, stream=stream)
    else:
        c.alltoall([t[o:] for t in src], [t[o:] for t in dst], count=n // k, dtype=hoc.UINT8, stream=stream)


def _sweep_footprint(op, n, k):
    """Bytes one op reads and writes (all ranks)."""
    return {"p2p": 2 * n, "allgather": n + k * n, "alltoall": 2 * k * n}[op]


def _sweep_verify(torch, op, src, dst, k, n):
    """Region 0 of the destinations holds exactly what the op must deliver."""
    if op == "p2p":
        return bool(torch.equal(dst[1][:n], src[0][:n]))
    cs = n // k
    for d in range(k):
        for r in range(k):
            want = src[r][:cs] if op == "allgather" else src[r][d * cs:(d + 1) * cs]
            if not torch.equal(dst[d][r * cs:(r + 1) * cs], want):
                return False
    return True


def leg_sweeps(sms):
    """Bandwidth vs size, 2 MB - 1 GB: copy engines vs TMA (all SMs, or 1/2/4/8 SMs).

    Sizes follow the nccl-tests convention of the paper's benchmarks: P2P = the
    message, AllGather = each rank's receive buffer, All-to-All = each rank's
    send buffer; algorithm bandwidth = size / time.  8 simulated ranks.  Each
    timed pass is one CUDA graph of back-to-back ops that cycle through
    regions of the rank buffers totalling >= 320 MB, so every op reads and
    writes HBM, not L2; the L2-warm figures (the same region every time) are
    separate rows for the sizes L2 can hold.  After timing, every point is
    run once more into zeroed destinations and checked byte for byte.
    """
    import torch

    from collective_communication_schedules_gb300 import hoc

    k = 8
    sizes_mb = [2, 8, 32, 128, 512, 1024]
    l2_sizes_mb = [2, 8, 32]
    variants = [("ce", 0), ("tma", 0), ("tma", 1), ("tma", 2), ("tma", 4), ("tma", 8)]
    big = max(sizes_mb) << 20
    g = torch.Generator(device="cuda").manual_seed(77)
    src = [torch.randint(0, 256, (big,), dtype=torch.uint8, device="cuda", generator=g) for _ in range(k)]
    dst = [torch.zeros(big, dtype=torch.uint8, device="cuda") for _ in range(k)]
    stream = torch.cuda.Stream()
    out = {"sizes_mb": sizes_mb, "l2": f"each timed pass cycles through >= {SWEEP_ROTATION_BYTES >> 20} MB of "
                                        "buffers (> 2x L2); the *_l2_warm rows reuse one region",
           "p2p": {}, "allgather": {}, "alltoall": {}, "regions_per_pass": {},
           "p2p_l2_warm": {}, "allgather_l2_warm": {}, "alltoall_l2_warm": {}, "l2_warm_sizes_mb": l2_sizes_mb,
           "verified": {}}

    def timed_graph(c, op, n, regions):
        with torch.cuda.stream(stream):
            for reg in sorted(set(regions)):                      # plans built outside the capture
                _sweep_call(c, hoc, op, src, dst, k, n, reg, stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for reg in regions:
                _sweep_call(c, hoc, op, src, dst, k, n, reg, stream)
        runs = []
        for i in range(4):                                        # one untimed replay, then the median of three
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                graph.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            if i:
                runs.append(e0.elapsed_time(e1))
        del graph
        return statistics.median(runs) / len(regions)

    for path, ctas in variants:
        name = path if ctas == 0 else f"{path}_{ctas}sm"
        c = hoc.Comm(k, torch.cuda.current_device(), hoc.Config(path=path, copy_max_sms=ctas))
        for op in ("p2p", "allgather", "alltoall"):
            row, warm, regs, ok = [], [], [], True
            for mb in sizes_mb:
                n = mb << 20
                nreg = max(1, min(big // n, -(-SWEEP_ROTATION_BYTES // _sweep_footprint(op, n, k))))
                reps = max(nreg, 3 if mb >= 512 else 10)
                ms = timed_graph(c, op, n, [i % nreg for i in range(reps)])
                row.append(round(n / (ms * 1e-3) / 1e9, 1))
                regs.append(nreg)
                if mb in l2_sizes_mb:
                    wms = timed_graph(c, op, n, [0] * 10)
                    warm.append(round(n / (wms * 1e-3) / 1e9, 1))
                with torch.cuda.stream(stream):                   # zeroed on the stream the op runs on
                    for t in dst:
                        t[:n].zero_()
                    _sweep_call(c, hoc, op, src, dst, k, n, 0, stream)
                torch.cuda.synchronize()
                ok = ok and _sweep_verify(torch, op, src, dst, k, n)
            out[op][name] = row
            out[op + "_l2_warm"][name] = warm
            out["regions_per_pass"].setdefault(op, regs)
            out["verified"].setdefault(op, {})[name] = ok
        c.close()
    del src, dst
    torch.cuda.empty_cache()
    return out


def leg_ce_allreduce_timeline(send, recv, k, local, stream, per_rank, peak):
    """When each chunk of the copy-engine allreduce is reduced and moved (the per-step timeline).

    One call with profiling on (events around every step), captured into a
    CUDA graph and replayed, after a few unprofiled calls.  Per chunk: the reduce kernel's start and end on the
    caller's stream, and the first start and last end of that chunk's copies
    over the copy queues.  Beside it, what the schedule's bytes cost at the
    measured copy rate: (3k - 1) S with no L2 reuse, 2kS if every all-gather
    read of a freshly reduced chunk hit L2.
    """
    import torch

    from collective_communication_schedules_gb300 import hoc

    out = {}
    for depth in (0, 2):
        with hoc.Comm(k, local, hoc.Config(path="ce", pipeline_depth=depth)) as c:
            for _ in range(3):
                c.allreduce(send, recv, stream=stream)
            ms = time_allreduce(c, send, recv, stream, 5)
            # The profiled call is captured into a CUDA graph (the library issues into the caller's
            # capture, the step events become graph nodes) and replayed: the same graph execution as
            # the library's own cached graphs, so the events do not change how the copies run.
            c.profile_enable(True)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                c.allreduce(send, recv, stream=stream)
            c.profile_enable(False)
            runs = []
            for _ in range(4):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                torch.cuda.synchronize()
                runs.append(e0.elapsed_time(e1))
            tl = c.profile_timeline()         # the events of the last replay
            del graph
        chunks = sorted({t["stage"] for t in tl})
        rows = []
        for q in chunks:
            red = [t for t in tl if t["stage"] == q and t["kind"] == "reduce"]
            mv = [t for t in tl if t["stage"] == q and t["kind"] == "copy"]
            rows.append({"chunk": q,
                         "reduce_ms": [round(red[0]["start_ms"], 4), round(red[0]["end_ms"], 4)] if red else None,
                         "moves_ms": [round(min(t["start_ms"] for t in mv), 4), round(max(t["end_ms"] for t in mv), 4)]
                         if mv else None})
        end = max(t["end_ms"] for t in tl)
        red_busy = sum(t["end_ms"] - t["start_ms"] for t in tl if t["kind"] == "reduce")
        out[f"depth_{depth or 'unbounded'}"] = {
            "ms_unprofiled": round(ms, 4), "ms_profiled_graph_replay": round(statistics.median(runs[1:]), 4),
            "timeline_end_ms": round(end, 4), "reduce_busy_ms": round(red_busy, 4), "chunks": rows}
    S = per_rank
    out["bytes_at_measured_copy_rate_ms"] = {
        "3k-1_S_no_l2_reuse": round((3 * k - 1) * S / (peak * 1e9) * 1e3, 4),
        "2kS_full_l2_reuse": round(2 * k * S / (peak * 1e9) * 1e3, 4)}
    return out


_SPIN = {}


def gpu_spin(stream, ms: float):
    """Queue a one-CTA FMA kernel that keeps `stream` busy for about `ms` ms, so that
    work the host queues behind it starts back to back, whatever the host's issue cost."""
    import torch

    from collective_communication_schedules_gb300 import hoc
    if "iters_per_ms" not in _SPIN:
        sink = torch.zeros(4, dtype=torch.float32, device="cuda")
        hoc.probe_launch(1, 32, 1000, stream=stream, sink=sink)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        hoc.probe_launch(1, 32, 20000, stream=stream, sink=sink)
        e1.record(stream)
        torch.cuda.synchronize()
        _SPIN["iters_per_ms"] = 20000 / max(e0.elapsed_time(e1), 1e-3)
        _SPIN["sink"] = sink
    hoc.probe_launch(1, 32, int(ms * _SPIN["iters_per_ms"]), stream=stream, sink=_SPIN["sink"])


def leg_startup_latency():
    """Time per copy of a chain of small copies on one stream, each waiting for the one before.

    HOCCL section 1 puts the DMA engines' startup latency at about 5x that of an
    SM-driven copy.  A chain of 100 copies of one size is queued behind a 3 ms
    spin kernel (so the host's issue cost is hidden) and timed with events
    around the chain: per copy = startup + transfer.  Copy engine vs the TMA
    kernel on 1 CTA and on every SM.
    """
    import torch

    from collective_communication_schedules_gb300 import hoc

    sizes = [4 << 10, 16 << 10, 64 << 10, 256 << 10, 1 << 20]
    chain = 100
    a = torch.randint(0, 256, (1 << 20,), dtype=torch.uint8, device="cuda")
    b = torch.zeros_like(a)
    stream = torch.cuda.Stream()
    out = {"sizes_bytes": sizes, "chain": chain, "us_per_copy": {}}
    for name, path, ctas in (("ce", "ce", 0), ("tma_1cta", "tma", 1), ("tma_all_sms", "tma", 0)):
        with hoc.Comm(2, torch.cuda.current_device(), hoc.Config(path=path, copy_max_sms=ctas)) as c:
            row = []
            for n in sizes:
                fn = lambda n=n: c.sendrecv(0, a, 1, b, n, hoc.UINT8, stream=stream)
                fn()
                torch.cuda.synchronize()
                runs = []
                for _ in range(3):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    gpu_spin(stream, 3.0)
                    e0.record(stream)
                    for _ in range(chain):
                        fn()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    runs.append(e0.elapsed_time(e1) * 1e3 / chain)
                row.append(round(statistics.median(runs), 3))
            out["us_per_copy"][name] = row
    ce, t1 = out["us_per_copy"]["ce"], out["us_per_copy"]["tma_1cta"]
    out["ce_over_tma_1cta"] = [round(x / y, 2) if y > 0 else None for x, y in zip(ce, t1)]
    out["ce_over_tma_all_sms"] = [round(x / y, 2) if y > 0 else None
                                  for x, y in zip(ce, out["us_per_copy"]["tma_all_sms"])]
    out["verified"] = bool(torch.equal(a, b))
    return out


def leg_host_overhead():
    """Host time of one call (CPU launch overhead, cf. Fig. 9), median over 200 calls."""
    import time as _t

    import torch

    from collective_communication_schedules_gb300 import hoc

    k, n = 8, 1 << 20
    a = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    b = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    g = [torch.empty(k * n, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    stream = torch.cuda.Stream()
    out = {}
    cases = {
        "allreduce_fused": ("fused", lambda c: c.allreduce(a, b, stream=stream)),
        "allreduce_ce_graph": ("ce", lambda c: c.allreduce(a, b, stream=stream)),
        "allgather_ce_graph": ("ce", lambda c: c.allgather(a, g, stream=stream)),
        "sendrecv_ce": ("ce", lambda c: c.sendrecv(0, a[0], 1, b[1], stream=stream)),
        "sendrecv_tma": ("tma", lambda c: c.sendrecv(0, a[0], 1, b[1], stream=stream)),
    }
    for name, (path, fn) in cases.items():
        with hoc.Comm(k, torch.cuda.current_device(), hoc.Config(path=path, chunk_bytes=1 << 18)) as c:
            fn(c)
            torch.cuda.synchronize()
            ts = []
            for i in range(200):
                t0 = _t.perf_counter()
                fn(c)
                ts.append((_t.perf_counter() - t0) * 1e6)
                if i % 20 == 19:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            out[name] = {"median_us": round(statistics.median(ts), 2), "p90_us": round(sorted(ts)[180], 2)}
    return out


def leg_paths_and_moves(args, send, recv, n_el, k, local, stream, sms, peak, per_rank):
    """Per-path allreduce figures with probes, the move half alone, copy size against interference,
    the chunk-size sweep and the allreduce under an SM budget."""
    import torch

    from collective_communication_schedules_gb300 import hoc

    # per-path figures
    paths = {}
    for p, eng in (("fused", "lsu"), ("fused", "tma"), ("ce", "lsu"), ("tma", "lsu")):
        c2 = hoc.Comm(k, local, hoc.Config(path=p, chunk_bytes=args.chunk_bytes, n_copy_streams=args.copy_streams,
                                           reduce_engine=eng))
        for _ in range(3):
            c2.allreduce(send, recv, stream=stream)
        pm = time_allreduce(c2, send, recv, stream, max(5, args.steps // 2))
        s2 = c2.last_stats()
        p = p if eng == "lsu" else f"{p}_{eng}"
        paths[p] = {"ms": round(pm, 4), "bus_gbs": round(bus_bytes(k, per_rank) / (pm * 1e-3) / 1e9, 1),
                    "hbm_frac": round(s2["bytes_exec"] / (pm * 1e-3) / (peak * 1e9), 4),
                    "lower_bound_frac": round(s2["bytes_min"] / (pm * 1e-3) / (peak * 1e9), 4),
                    "sms_used": s2["sms_used"], "kernels_per_step": s2["kernels"],
                    "copies_per_step": s2["copies"]}
        paths[p]["probe"] = probes(lambda s, c2=c2: c2.allreduce(send, recv, stream=s), pm, stream, sms)
        c2.close()
    # the move half alone: all-gather of the 32 MiB blocks, copy engines vs TMA
    ag = {}
    blk = n_el // k
    ag_send = [t[:blk] for t in send]
    for p in ("ce", "tma"):
        c3 = hoc.Comm(k, local, hoc.Config(path=p, chunk_bytes=args.chunk_bytes, n_copy_streams=args.copy_streams))
        run = lambda s, c3=c3: c3.allgather(ag_send, recv, stream=s)
        for _ in range(3):
            run(stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            run(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        am = e0.elapsed_time(e1) / 10
        s3 = c3.last_stats()
        ag[p] = {"ms": round(am, 4), "bytes_gbs": round(s3["bytes_exec"] / (am * 1e-3) / 1e9, 1),
                 "sms_used": s3["sms_used"], "kernels_per_step": s3["kernels"],
                 "probe": probes(run, am, stream, sms),
                 # the same probe train on a stream of the highest priority (the moves' streams keep
                 # the default, lowest one): compute first wherever the GPU arbitrates between streams
                 "probe_high_priority": probes(run, am, stream, sms, priority=-100),
                 # the same train at default priority, each kernel launched with programmatic dependent
                 # launch: the launch overlaps the kernel before it
                 "probe_pdl": probes(run, am, stream, sms, pdl=True)}
        c3.close()
    # copy-engine chunk size against interference: larger copies move faster but slow the probe more
    tradeoff = []
    for mib, nq in ((4, 4), (8, 4), (16, 4), (32, 4), (32, 8)):
        c5 = hoc.Comm(k, local, hoc.Config(path="ce", chunk_bytes=mib << 20, n_copy_streams=nq))
        run = lambda s, c5=c5: c5.allgather(ag_send, recv, stream=s)
        for _ in range(3):
            run(stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            run(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        am = e0.elapsed_time(e1) / 10
        s5 = c5.last_stats()
        pr = probes(run, am, stream, sms)
        tradeoff.append({"chunk_mib": mib, "copy_streams": nq, "ms": round(am, 4),
                         "bytes_gbs": round(s5["bytes_exec"] / (am * 1e-3) / 1e9, 1), "copies_per_step": s5["copies"],
                         "kernels_per_step": s5["kernels"],
                         "probe_slowdown": {sh: pr[sh]["slowdown"] for sh in pr},
                         "probe_sm_mhz_with": {sh: pr[sh]["sm_mhz_with"] for sh in pr}})
        c5.close()
    out = {"paths": paths, "allgather_moves": ag, "allgather_ce_chunk_vs_probe": tradeoff}
    # chunk size sweep, 1-64 MiB (64 is capped at the 32 MiB block), on the copy-engine and
    # TMA-kernel move paths; then copy-queue counts on the copy-engine path
    sweep = []
    grid = [(p, mib, 4, 0) for p in ("ce", "tma") for mib in (1, 2, 4, 8, 16, 32, 64)]
    grid += [("ce", 32, 8, 0), ("ce", 8, 8, 0), ("ce", 8, 16, 0)]
    grid += [("ce", 4, 4, d) for d in (1, 2, 4)]      # pipeline depth: reduce at most d chunks ahead of the moves
    for p, chunk_mib, nq, depth in grid:
        c4 = hoc.Comm(k, local, hoc.Config(path=p, chunk_bytes=chunk_mib << 20, n_copy_streams=nq,
                                           pipeline_depth=depth))
        for _ in range(3):
            c4.allreduce(send, recv, stream=stream)
        cm = time_allreduce(c4, send, recv, stream, 10)
        s4 = c4.last_stats()
        sweep.append({"path": p, "chunk_mib": chunk_mib, "copy_streams": nq, "pipeline_depth": depth or "unbounded",
                      "ms": round(cm, 4),
                      "bus_gbs": round(bus_bytes(k, per_rank) / (cm * 1e-3) / 1e9, 1),
                      "lower_bound_frac": round(s4["bytes_min"] / (cm * 1e-3) / (peak * 1e9), 4),
                      "copies_per_step": s4["copies"], "kernels_per_step": s4["kernels"]})
        c4.close()
    out["chunk_sweep"] = sweep
    # allreduce under an SM budget: fused (every move on the few SMs) vs copy engines (SMs only reduce);
    # AUTO picks the copy engines when a budget is set
    budget = []
    for m in (8, 32):
        for p in ("fused", "ce"):
            c6 = hoc.Comm(k, local, hoc.Config(path=p, reduce_max_sms=m))
            for _ in range(2):
                c6.allreduce(send, recv, stream=stream)
            bm = time_allreduce(c6, send, recv, stream, 5)
            s6 = c6.last_stats()
            budget.append({"reduce_max_sms": m, "path": p, "ms": round(bm, 3),
                           "bus_gbs": round(bus_bytes(k, per_rank) / (bm * 1e-3) / 1e9, 1),
                           "sms_used": s6["sms_used"], "copies_per_step": s6["copies"]})
            c6.close()
    out["allreduce_under_sm_budget"] = budget
    return out


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    n_el = args.count
    xs_host = generate_inputs(K_RANKS, n_el)    # spawned workers, before the first CUDA call
    bucket_pool = None
    if args.workloads and not args.no_extras:
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        with ProcessPoolExecutor(max_workers=min(16, os.cpu_count() or 1), mp_context=mp.get_context("spawn")) as ex:
            bucket_pool = list(ex.map(_gen_bucket, [(s_, r_) for s_ in range(16) for r_ in range(K_RANKS)]))
    from collective_communication_schedules_gb300 import hoc

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sms = hoc.sm_count(local)
    peak, peak_kind = measured_peaks()
    per_rank = n_el * 2
    k = K_RANKS
    h_send = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs_host]
    h_recv = [torch.empty_like(t).pin_memory() for t in h_send]
    send = [t.to(dev) for t in h_send]
    recv = [torch.empty_like(t) for t in send]
    stream = torch.cuda.Stream(device=dev)
    cfg = hoc.Config(path=args.path, chunk_bytes=args.chunk_bytes, n_copy_streams=args.copy_streams)
    comm = hoc.Comm(k, local, cfg)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            comm.allreduce(send, recv, stream=stream)
    torch.cuda.synchronize()
    st = comm.last_stats()
    fused = st["path"] == hoc.PATH_FUSED
    kernel_kind = hoc.KERNEL_FUSED if fused else hoc.KERNEL_REDUCE

    # ---- timed region (device events on the launching stream; inputs 2 GiB > L2)
    sampler = ClockSampler(gpu_id_for(local))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    if fused:
        comm.profile_enable(True)      # one launch per step, no graph: events bracket the kernel itself
    ms = time_allreduce(comm, send, recv, stream, args.steps)
    clocks = sampler.stop()
    torch.cuda.synchronize()
    barrier(world)
    if not fused:
        comm.profile_enable(True)      # graphs are off while profiling: a separate pass of the same steps
        time_allreduce(comm, send, recv, stream, args.steps)
    launches, kern_ms = comm.profile_read(kernel_kind)
    comm.profile_enable(False)
    ms_max = max_over_ranks(world, ms, dev)
    busbw = bus_bytes(k, per_rank) / (ms_max * 1e-3) / 1e9
    value = world * busbw
    st = comm.last_stats()
    hbm_frac = st["bytes_exec"] / (ms_max * 1e-3) / (peak * 1e9)
    lb_frac = st["bytes_min"] / (ms_max * 1e-3) / (peak * 1e9)
    # algorithmic bytes of the dominant kernel per launch
    if fused:
        kern_bytes = 2 * k * per_rank
        kname = "fused_reduce_broadcast"
    else:
        launches_per_step = max(1, launches // max(1, args.steps))
        kern_bytes = (k + 1) * per_rank // launches_per_step
        kname = "reduce"
    avg_launch_ms = kern_ms / max(1, launches)
    achieved = kern_bytes / (avg_launch_ms * 1e-3) / 1e9 if launches else None
    roofline = {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1) if achieved else None,
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4) if achieved else None,
                "traffic": recorded_traffic(kname, k, n_el), "bytes_per_launch": kern_bytes,
                "avg_launch_ms": round(avg_launch_ms, 4), "launches": launches,
                "peak_source": f"{peak_kind}: MEASURED_PEAKS.json hbm_gbs, the copy rate a STREAM-style copy reaches "
                               "on this GPU (an empirical ceiling, which a kernel can slightly exceed)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4) if achieved else None}

    # ---- end to end: pinned host inputs -> device, allreduce, results -> host
    # End to end through the host-buffer call: every step brings the 2 GiB of
    # inputs in from pinned host memory and the 2 GiB of results out.  With
    # path AUTO the call runs directly on the host buffers (one fused launch
    # whose loads and stores cross the host link); the staged copy-engine
    # pipeline (path CE) is timed beside it.
    def time_host(c):
        c.allreduce_host(h_send, h_recv, stream=stream)         # untimed: first touch, graph capture
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            c.allreduce_host(h_send, h_recv, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.e2e_steps, c.last_stats()
    e2e_ms, e2e_st = time_host(comm)
    e2e_ms = max_over_ranks(world, e2e_ms, dev)
    with hoc.Comm(k, local, hoc.Config(path="ce")) as c_ce:
        staged_ms, staged_st = time_host(c_ce)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the same step done the plain way: all inputs in, allreduce, all results out
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(args.e2e_steps):
            for r in range(k):
                send[r].copy_(h_send[r], non_blocking=True)
            comm.allreduce(send, recv, stream=stream)
            for r in range(k):
                h_recv[r].copy_(recv[r], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    plain_ms = e0.elapsed_time(e1) / args.e2e_steps
    mode = "direct: one fused launch on the pinned host buffers" if e2e_st["copies"] == 0 else \
        "staged: copy-engine pipeline through device slots"
    e2e = {"value": round(world * bus_bytes(k, per_rank) / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": k * per_rank, "d2h_bytes_per_step": k * per_rank, "ms_per_step": round(e2e_ms, 3),
           "call": f"hoc_allreduce_host, path {args.path} ({mode})",
           "staged_ce_ms_per_step": round(staged_ms, 3), "staged_ce_copies_per_step": staged_st["copies"],
           "unpipelined_ms_per_step": round(plain_ms, 3)}

    extras = {}

    def study(fn, *a):
        """Run one study leg; a leg that fails is reported in the line and the headline stands."""
        try:
            return fn(*a)
        except Exception as e:  # noqa: BLE001 -- any failure of a study leg is data for the line
            try:
                torch.cuda.synchronize()
                torch.cuda.empty_cache()
            except Exception:  # noqa: BLE001
                pass
            return {"error": f"{type(e).__name__}: {e}"}

    if not args.no_extras:
        pm = study(leg_paths_and_moves, args, send, recv, n_el, k, local, stream, sms, peak, per_rank)
        if "error" in pm:
            extras["paths_and_moves"] = pm
        else:
            extras.update(pm)
        extras["ce_interference"] = study(leg_ce_interference, send, recv, n_el, k, local, stream, sms)
        extras["ce_allreduce_timeline"] = study(leg_ce_allreduce_timeline, send, recv, k, local, stream, per_rank,
                                                peak)
    if args.workloads and not args.no_extras:
        extras["workloads"] = {"dp_bucket_stream": study(leg_bucket_stream, bucket_pool, sms, peak),
                               "pp_1f1b": study(leg_pipeline, sms),
                               "ep_dispatch_combine": study(leg_expert_dispatch, peak)}
        if isinstance(extras["workloads"]["dp_bucket_stream"], dict):
            extras["workloads"]["dp_bucket_stream"]["cpu_baseline"] = study(cpu_baseline_buckets, bucket_pool)
        bucket_pool = None
        extras["sweeps"] = study(leg_sweeps, sms)
        extras["startup_latency"] = study(leg_startup_latency)
        extras["host_overhead_us"] = study(leg_host_overhead)

    cpu = None
    if rank == 0:
        cpu = cpu_baseline(xs_host, args.cpu_seconds, device_out=recv)
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": oracle_config() if n_el == N_ELEMS else
                {"workload": f"profiling case: 8 ranks x {n_el:,} bf16", "k": k, "count": n_el},
                "schedule": {"path": args.path,
                             "resolved_path": {0: "auto", 1: "ce", 2: "tma", 3: "fused"}[st["path"]],
                             "chunk_bytes": args.chunk_bytes or "auto (by move path and rank count; 4 MiB at 8 ranks)",
                             "copy_streams": args.copy_streams or "auto (8 for copies of at most 2 MiB, else 4)"},
                "algbw_gbs": round(per_rank / (ms_max * 1e-3) / 1e9, 2),
                "hbm_frac": round(hbm_frac, 4), "lower_bound_frac": round(lb_frac, 4),
                "sms_used": st["sms_used"], "gpu_launches": st["kernels"] * args.steps,
                "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks}
        line.update(extras)
        print(json.dumps(line), flush=True)
    comm.close()


def run_allgather_only(args, world, rank, local):
    """The move half alone: 8 ranks x 32 MiB blocks gathered to every rank."""
    import torch

    from collective_communication_schedules_gb300 import hoc

    torch.cuda.set_device(local)
    k, blk = K_RANKS, args.count // K_RANKS
    g = torch.Generator(device="cuda").manual_seed(2)
    send = [torch.randn(blk, generator=g, device="cuda").to(torch.bfloat16) for _ in range(k)]
    recv = [torch.empty(k * blk, dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    stream = torch.cuda.Stream()
    with hoc.Comm(k, local, hoc.Config(path=args.path if args.path != "fused" else "ce",
                                       chunk_bytes=args.chunk_bytes, n_copy_streams=args.copy_streams)) as c:
        for _ in range(args.warmup):
            c.allgather(send, recv, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            c.allgather(send, recv, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        st = c.last_stats()
    if rank == 0:
        print(json.dumps({"metric": "simulated-rank allgather moved GB/s (profiling case)", "unit": "GB/s",
                          "value": round(st["bytes_exec"] / (ms * 1e-3) / 1e9, 1), "ms_per_step": round(ms, 4),
                          "steps": args.steps, "path": args.path, "kernels_per_step": st["kernels"],
                          "copies_per_step": st["copies"], "sms_used": st["sms_used"]}), flush=True)


def run_ep_fused_only(args, world, rank, local):
    """The EP round trip fused with the exchange alone (a profiling case): dispatch + combine."""
    import numpy as np
    import torch

    from collective_communication_schedules_gb300 import hoc, inputs

    torch.cuda.set_device(local)
    w = inputs.EP_DISPATCH
    k, tokens, h, experts, topk = w["k"], w["tokens"], w["hidden"], w["experts"], w["topk"]
    routing = inputs.ep_routing(k, tokens, experts, topk, w["zipf"])
    g = torch.Generator(device="cuda").manual_seed(5500)
    xs = [torch.randn((tokens, h), generator=g, device="cuda").to(torch.bfloat16) for _ in range(k)]
    ids = [torch.from_numpy(routing[r].astype(np.int32).reshape(-1)).cuda() for r in range(k)]
    gate = [torch.rand(tokens * topk, generator=g, device="cuda") for _ in range(k)]
    cnt = np.stack([np.bincount(routing[r].reshape(-1) // (experts // k), minlength=k) for r in range(k)])
    cap = [int(cnt[:, d].sum()) * h for d in range(k)]
    recv = [torch.empty(cap[d], dtype=torch.bfloat16, device="cuda") for d in range(k)]
    pos = [torch.empty(tokens * topk, dtype=torch.int32, device="cuda") for _ in range(k)]
    counts = torch.empty((k, k), dtype=torch.int64, device="cuda")
    wsp = torch.empty(k * hoc.ep_pack_workspace(tokens, topk, experts), dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = [torch.empty((tokens, h), dtype=torch.bfloat16, device="cuda") for _ in range(k)]
    stream = torch.cuda.Stream()

    def step():
        hoc.ep_dispatch_fused(ids, xs, experts, recv, cap, pos, counts, wsp, status, stream=stream)
        hoc.ep_combine_fused(recv, cap, ids, pos, counts, gate, tokens, topk, h, experts, ys, status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    ph = []
    for _ in range(args.steps):   # the two phases apart, each between events
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        hoc.ep_dispatch_fused(ids, xs, experts, recv, cap, pos, counts, wsp, status, stream=stream)
        ev[1].record(stream)
        hoc.ep_combine_fused(recv, cap, ids, pos, counts, gate, tokens, topk, h, experts, ys, status, stream=stream)
        ev[2].record(stream)
        torch.cuda.synchronize()
        ph.append((ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])))
    if rank == 0:
        print(json.dumps({"metric": "EP dispatch + combine fused with the exchange (profiling case)", "unit": "ms",
                          "value": round(ms, 4), "steps": args.steps, "status": int(status.item()),
                          "dispatch_ms": round(statistics.median(p[0] for p in ph), 4),
                          "combine_ms": round(statistics.median(p[1] for p in ph), 4),
                          "config": {"k": k, "tokens": tokens, "hidden": h, "experts": experts, "topk": topk}}),
              flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()
    if world > 1:
        # N replicas: the timed region and the end-to-end leg run on every rank (max over ranks); the
        # per-path, probe, sweep and workload legs are single-GPU studies and run at N = 1 only
        args.no_extras = True
    if args.mode == "allgather":
        run_allgather_only(args, world, rank, local)
    elif args.mode == "ep_fused":
        run_ep_fused_only(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
