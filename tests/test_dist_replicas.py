"""Multi-process plumbing of bench.py on CPU (gloo, world size 2): the path
shards as independent replicas, so the only cross-rank steps are the barrier
around the timed region and the max over ranks of the elapsed time."""
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


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r "took" (r + 1) * 10 ms: every rank must see the slowest
        t = bench.all_max(10.0 * (rank + 1), world)
        results[rank] = (t, bench.aggregate_gbs(world, 4 * 10**9, t))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 20.0
    # two replicas of a 4 GB step in 20 ms -> 400 GB/s for the job
    assert res[0][1] == pytest.approx(400.0)


def test_single_process_aggregate_is_plain_throughput():
    import bench
    assert bench.aggregate_gbs(1, 330_272_620, 0.05) == pytest.approx(6605.4524)
    assert bench.all_max(3.0, 1) == 3.0
