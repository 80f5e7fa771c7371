"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): each rank prefills its
own pack (weak scaling, no collective on the data path); the job's time is the slowest
rank's and its throughput counts every rank's tokens."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier(world)
    ms_local = 10.0 + 5.0 * rank          # rank 1 is the slow one
    ms, value = bench.aggregate(32768, ms_local, world)
    results[rank] = (ms, value)
    bench.barrier(world)
    dist.destroy_process_group()


def test_weak_scaling_aggregate_two_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        ms, value = results[r]
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(32768 * 2 / 0.015)


def test_single_rank_aggregate_is_local():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(32768, 2.0, 1)
    assert ms == 2.0 and value == pytest.approx(32768 / 0.002)
