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
