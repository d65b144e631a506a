"""bench.py's multi-rank reduction on CPU: two gloo ranks, max-over-ranks
timing, whole-job throughput = all ranks' units over the slowest rank."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = 0.5 if rank == 0 else 2.0  # rank 1 is the slow one
    value, slowest = bench.aggregate(units_per_rank=64, rank_seconds=seconds, world=world)
    results[rank] = (value, slowest, bench.dist_env())
    dist.destroy_process_group()


def test_aggregate_uses_slowest_rank():
    world = 2
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        value, slowest, env = res[rank]
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(64 * world / 2.0)
        assert env == (world, rank, rank)


def test_single_rank_is_identity():
    import bench
    value, slowest = bench.aggregate(units_per_rank=10, rank_seconds=0.25, world=1)
    assert slowest == 0.25 and value == pytest.approx(40.0)
