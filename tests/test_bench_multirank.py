"""bench.py's multi-rank host logic on CPU: two gloo ranks (one replica each,
weak scaling) agree on the max time and the summed work over ranks."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_env() == (rank, world, rank)
        t = bench.max_over_ranks(1.5 + rank)       # each rank's own step time
        w = bench.sum_over_ranks(1000.0 * (rank + 1))  # each rank's processed bytes
        bench.barrier()
        results[rank] = (t, w)
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions_over_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    assert dict(results) == {0: (2.5, 3000.0), 1: (2.5, 3000.0)}


def test_single_process_reductions_are_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.sum_over_ranks(7.0) == 7.0
    bench.barrier()
