"""The replica (N > 1) path of bench.py on CPU: two gloo ranks combine their
step times. The job's step time is the slowest rank's, and the throughput
counts every rank's bytes."""

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


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    step_bytes = 1.0e9
    ms, gbs = bench._aggregate(step_bytes, 1.0 + rank, world, dist, "cpu")  # rank 1 is slower
    out[rank] = (ms, gbs, bench._max_over_ranks(-rank, dist, "cpu"))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        ms, gbs, mx = out[rank]
        assert ms == 2.0                       # the slower rank's step time
        assert gbs == pytest.approx(world * 1.0e9 / 2.0e-3 / 1e9)
        assert mx == 0.0                       # max(-0, -1)


def test_single_process_is_local():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._aggregate(2.0e9, 4.0, 1, None, "cpu") == (4.0, pytest.approx(500.0))
