"""The multi-rank (replica) path of the benchmark on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own copy of the workload; the job's time is the slowest rank's, and the
throughput counts every rank's units over that time (weak scaling).  No data-path collective
exists: only this timing reduction crosses ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, local_ms, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        slowest = bench.max_over_ranks(local_ms[rank])
        results[rank] = (env, slowest, bench.replica_throughput(1000, slowest, world))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_replicas_time_is_the_slowest_rank():
    world, local_ms = 2, [12.5, 20.0]
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_worker, args=(world, _free_port(), local_ms, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        env, slowest, tput = res[rank]
        assert env == (rank, world, rank)
        assert slowest == 20.0
        # 2 ranks x 1000 units in 20 ms
        assert tput == pytest.approx(2 * 1000 / 0.020)


def test_single_rank_throughput_is_units_over_time():
    assert bench.replica_throughput(8192 * 20, 15.0, 1) == pytest.approx(8192 * 20 / 0.015)
