"""The N-rank aggregation of bench.py on CPU with two gloo ranks: every rank
gets the slowest rank's step time and the whole-job throughput."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.aggregate(1.0 + rank * 0.5, 1000, world, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == pytest.approx(1.5)
        assert value == pytest.approx(world * 1000 / 1.5e-3)


def test_single_rank_is_local():
    import bench
    assert bench.aggregate(2.0, 500, 1) == (2.0, 500 / 2e-3)
