"""CPU oracle for the HOCCL collective schedules -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the collectives compute,
written in numpy.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
CUDA library never imports, links or calls anything here, and nothing here
imports the CUDA library: the two share only the seeded input generators.

Sources (HOCCL: Offloading Collective Communication from GPU Cores to
Accelerate Distributed Training):
  * section 5 (Limitations): reductions (AllReduce, ReduceScatter) are outside
    the paper's zero-SM scope, so their arithmetic is fixed here by the
    textbook ring convention (oracle.ring);
  * section 6.2 (Communication Benchmark), "AllGather" / "All-to-All":
    semantics of the move-only collectives (oracle.ring.allgather,
    oracle.alltoall);
  * section 3.4 (Collective Scheduler), Eq. 6-8: stage decomposition
    invariants (oracle.alltoall.shift_stages);
  * section 2.1 (Distributed Training Workloads): PP send/recv overlapped
    with compute (oracle.pipeline).

Modules
-------
bf16      -- bfloat16 <-> binary32 conversions from the IEEE definition.
exact     -- exact rational arithmetic and correctly rounded binary32, used only
             by the pins in tests/.
ring      -- ring reduce-scatter / allreduce fold, allgather.
alltoall  -- all-to-all(v), shift stages.
pipeline  -- 1F1B schedule and the PP XOR workload.

Parity status: every function has at least one pin in tests/test_oracle_*.py
except the choice of ring order itself (any permutation is a valid ring);
parity is defined given the ring order.  Parity unpinned: ring order choice.
"""
from . import bf16, ring, alltoall, pipeline, exact  # noqa: F401
