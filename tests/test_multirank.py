"""Multi-rank bookkeeping of bench.py on CPU: world size 2 over gloo.

Every rank runs an independent replica (no collective on the data path); the
only cross-rank steps are a barrier and the max / sum reductions of the timing
and of the bytes processed, which these tests exercise.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench._dist_env()
        assert (ws, r, local) == (world, rank, rank)
        bench.barrier()
        slowest = bench.reduce_over_ranks(1.5 + rank, "max")
        total = bench.reduce_over_ranks(10.0 * (rank + 1), "sum")
        results[rank] = (slowest, total)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_sum():
    world = 2
    port = _free_port()
    with mp.Manager() as manager:
        results = manager.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        got = dict(results)
    for rank in range(world):
        assert got[rank] == (2.5, 30.0)


def test_single_process_reductions_are_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.reduce_over_ranks(3.25, "max") == 3.25
    assert bench.reduce_over_ranks(3.25, "sum") == 3.25
    bench.barrier()
