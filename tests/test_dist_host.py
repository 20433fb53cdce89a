"""The bench's multi-replica host logic on CPU: world size 2 over gloo.

Each replica times its own work; rank 0 reports the maximum over ranks and
the whole-job value scales with the number of replicas.
"""
import os
import socket

import torch.multiprocessing as tmp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), HOC_DIST_BACKEND="gloo")
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    mine = 1.5 + rank            # this replica's step time (ms)
    out[rank] = bench.max_over_ranks(w, mine)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_max_time():
    world, port = 2, _free_port()
    mgr = tmp.Manager()
    out = mgr.dict()
    tmp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_bus_bytes_convention():
    import bench
    # nccl-tests bus bandwidth factor for allreduce: 2(k-1)/k
    assert bench.bus_bytes(8, 256 << 20) == 2 * 7 / 8 * (256 << 20)
    assert bench.bus_bytes(1, 100) == 0


def test_reference_arm_under_torchrun_prints_one_line():
    """`bench.py --impl reference` launched as two replicas: rank 0 alone times the oracle and prints one
    JSON line; the other rank exits 0 without work (CPU, gloo)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, HOC_DIST_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same workload description and the same oracle sample as the GPU arm's cpu_baseline
    import bench
    assert d["config"] == bench.oracle_config()
    assert d["cpu_baseline"]["sample"].startswith(bench.cpu_sample_text().split(";")[0])
