"""The benchmark's multi-rank aggregation on CPU: two gloo ranks (no GPU).

Each rank encodes its own workload (independent problems, no data-path
collective); the job time is the slowest rank's, and the whole-job rate is
the units of all ranks over that time.
"""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # rank r took (r + 1) ms per step and (10 - r) s of region time
        kernel_ms, region_s = bench.reduce_max([rank + 1.0, 10.0 - rank], "cpu")
        results[rank] = (kernel_ms, region_s,
                         bench.job_throughput(1000.0, world, kernel_ms * 1e-3))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    with mp.Manager() as manager:
        results = manager.dict()
        mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world,
                           start_method="spawn")
        got = dict(results)
    for rank in range(world):
        kernel_ms, region_s, rate = got[rank]
        assert kernel_ms == 2.0  # the slower rank's step time
        assert region_s == 10.0
        assert rate == 1000.0 * world / 2e-3


def test_single_process_is_identity():
    assert bench.reduce_max([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
