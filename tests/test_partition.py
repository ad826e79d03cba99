"""The multi-GPU partition of one encode job (``vq_partition``).

Every sub-vector is encoded on its own against its group's codebook, so one
job ``[G][M]`` splits across ranks with no exchange: each rank owns a
balanced contiguous range of the flattened rows, encodes it against the
replicated codebooks as at most three grouped encodes, and keeps its indices.

CPU (no GPU): the partition owns every row exactly once, in row order, for
ragged and degenerate sizes; and two ``gloo`` ranks each take their slices,
encode them (the oracle as the encoder), gather them and reassemble the
whole-job oracle result bit for bit.  GPU: the ranks' shares, encoded by the
library one rank after another on one device, concatenate to the whole-job
encode.
"""
import ctypes
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


@pytest.fixture(scope="module")
def vq():
    from product_vq_kv_gb300.build import build

    build()
    import product_vq_kv_gb300 as m

    m.load_library()
    return m


SIZES = [(1, 1), (1, 7), (3, 10), (5, 7), (2, 128 * 3 + 5), (7, 1), (256, 513), (0, 5), (4, 0),
         (1, 1 << 20), (3, (1 << 31) + 5)]


@pytest.mark.parametrize("g,m", SIZES)
@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8])
def test_every_row_owned_exactly_once(vq, g, m, world):
    total = g * m
    shares, prev_end = [], 0
    for rank in range(world):
        slices = vq.vq_partition(g, m, world, rank)
        assert len(slices) <= 3
        n = 0
        for g0, ng, r0, nr in slices:
            assert ng >= 1 and nr >= 1 and 0 <= g0 and g0 + ng <= g and 0 <= r0 and r0 + nr <= m
            if ng > 1:
                assert r0 == 0 and nr == m  # whole groups
            first = g0 * m + r0
            # contiguous, in row order: each slice starts where the last ended
            assert first == prev_end
            prev_end = (g0 + ng - 1) * m + r0 + nr
            n += ng * nr
        shares.append(n)
    assert prev_end == total and sum(shares) == total
    assert max(shares) - min(shares) <= 1
    # the share sizes are floor((r + 1) T / world) - floor(r T / world)
    assert shares == [(r + 1) * total // world - r * total // world for r in range(world)]


def test_partition_rejects_bad_arguments(vq):
    import product_vq_kv_gb300._binding as b

    lib = vq.load_library()
    buf = (b.VqSlice * 3)()
    n = ctypes.c_int32(0)
    for args in [(2, 5, 0, 0), (2, 5, 2, 2), (2, 5, 2, -1), (-1, 5, 1, 0), (2, -5, 1, 0),
                 (1 << 40, 1 << 40, 1, 0)]:
        assert lib.vq_partition(*args, buf, ctypes.byref(n)) == vq.VQ_ERR_INVALID_ARG, args
    assert lib.vq_partition(2, 5, 1, 0, None, ctypes.byref(n)) == vq.VQ_ERR_INVALID_ARG
    assert lib.vq_partition(2, 5, 1, 0, buf, None) == vq.VQ_ERR_INVALID_ARG


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _job(seed=5, g=3, m=1000, sub=8, n_c=256):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((g, m, sub)).astype(np.float16)
    cb = rng.standard_normal((g, n_c, sub)).astype(np.float16)
    return x, cb


def _rank(rank: int, world: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        import product_vq_kv_gb300 as vq

        x, cb = _job()  # every rank holds the job's inputs; codebooks replicated
        parts = []
        for g0, ng, r0, nr in vq.vq_partition(x.shape[0], x.shape[1], world, rank):
            parts.append(oracle.encode(np.ascontiguousarray(x[g0:g0 + ng, r0:r0 + nr]),
                                       np.ascontiguousarray(cb[g0:g0 + ng])).reshape(-1))
        mine = np.concatenate(parts) if parts else np.zeros(0, np.uint32)
        gathered = [None] * world
        dist.all_gather_object(gathered, mine)
        if rank == 0:
            whole = np.concatenate(gathered)
            results["equal"] = bool(np.array_equal(whole, oracle.encode(x, cb).reshape(-1)))
            results["sizes"] = [int(a.size) for a in gathered]
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reassemble_the_whole_job(vq, oracle_mod):
    world = 2
    with mp.Manager() as manager:
        results = manager.dict()
        mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world,
                           start_method="spawn")
        got = dict(results)
    assert got["equal"]
    assert got["sizes"] == [1500, 1500]


@pytest.mark.gpu
@pytest.mark.parametrize("world", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("g,m", [(3, 1000), (32, 8192), (1, 128 * 9 + 7)])
def test_shares_concatenate_to_the_whole_encode(vq, oracle_mod, world, g, m):
    x, cb = _job(seed=world + m, g=g, m=m)
    xd, cbd = torch.from_numpy(x).cuda(), torch.from_numpy(cb).cuda()
    whole = vq.vq_encode_grouped(xd, cbd).reshape(-1)
    shares = [vq.vq_encode_partition(xd, cbd, world, rank) for rank in range(world)]
    got = torch.cat([s.view(torch.int32) for s in shares])
    assert torch.equal(got, whole.view(torch.int32))
    want = oracle_mod.encode(x, cb, n_threads=os.cpu_count() or 1).reshape(-1)
    assert np.array_equal(got.cpu().numpy().view(np.uint32), want)
