"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each a replica of
independent work (weak scaling, no data-path collective); the job time is the
slowest rank's and the throughput counts every rank's units."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world, device="cpu")
    thr = bench.job_throughput(8192, ms, world, device="cpu")
    bench.barrier(world)
    results[rank] = (worst, thr)
    dist.destroy_process_group()


def test_two_rank_weak_scaling_reduction():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        worst, thr = res[rank]
        assert worst == pytest.approx(5.0)
        assert thr == pytest.approx(8192 * 2 / 5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.0, 1) == 4.0
    assert bench.job_throughput(100, 10.0, 1) == pytest.approx(100 / 1e-2)
