"""Multi-process host logic of bench.py (CPU, gloo, world size 2): the barrier and the
max-over-ranks timing, and the whole-job throughput of independent replicas."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        assert (r, w, lr) == (rank, world, rank)
        bench.barrier(w)
        ms = [12.5, 20.0][rank]                     # rank 1 is the slowest
        ms_max = bench.max_over_ranks(ms, w)
        out[rank] = ms_max
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_replica_throughput_counts_all_ranks_at_the_slowest_time():
    # 2 replicas x batch 4 x 100 steps in 0.5 s (slowest rank) -> 1,600 tok/s
    assert bench.replica_throughput(2, 4, 100, 500.0) == pytest.approx(1600.0)
    assert bench.replica_throughput(1, 1, 511, 1000.0) == pytest.approx(511.0)
