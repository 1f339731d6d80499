"""The N > 1 path of bench.py (independent replicas) on CPU with gloo, world size 2.

The path does not shard: each rank runs the whole workload on its own GPU and the
only cross-rank step is the timing reduction -- max of the elapsed times, sum of
the units processed.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, 0)
        elapsed = 1.0 + rank  # rank 1 is the slowest
        units = 10.0 * (rank + 1)
        results[rank] = bench.replica_reduce(elapsed, units, world)
    finally:
        dist.destroy_process_group()


def test_replica_reduce_two_ranks():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        for r in range(2):
            assert results[r] == (2.0, 30.0)  # max elapsed, summed units, identical on every rank


def test_single_rank_is_identity():
    import bench
    assert bench.replica_reduce(3.5, 7.0, 1) == (3.5, 7.0)
