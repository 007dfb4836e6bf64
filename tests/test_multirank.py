"""The N>1 path of bench.py on CPU: two gloo ranks, each with its own batch
(weak scaling, no collective on the data), timing reduced by max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        class A:
            workload = "tiny"
            Ls = None
            seed = 5
        case = bench.build_case(A, rank)
        # each rank times its own batch; the job time is the slowest rank
        local_ms = 1.0 + rank
        t = bench.max_over_ranks(local_ms, world)
        bench.barrier(world)
        out[rank] = (t, float(case.q.float().sum()), case.total_q())
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    t0, q0, rows0 = out[0]
    t1, q1, rows1 = out[1]
    assert t0 == t1 == 2.0                 # max over ranks, seen by every rank
    assert q0 != q1                        # independent batches (seed + rank)
    assert rows0 == rows1 == 4             # same work per rank: weak scaling


def test_reference_arm_other_ranks_exit(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        pass
    assert bench.run_reference(A) == 0     # rank != 0: no work, exit 0
