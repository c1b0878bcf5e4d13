"""The weak-scaling aggregation of bench.py across ranks (gloo, two processes on the CPU):
the whole job's time is the slowest rank's and its bytes are the sum over ranks."""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    maxima, sums = bench.reduce_over_ranks(torch, "cpu", [1.0 + rank, 10.0 * (rank + 1)],
                                           [100.0 * (rank + 1), 7.0])
    queue.put((rank, maxima, sums))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, maxima, sums in results:
        assert maxima == [2.0, 20.0]
        assert sums == [300.0, 14.0]


def test_reduce_single_process_passes_through():
    torch = pytest.importorskip("torch")
    import bench

    assert bench.reduce_over_ranks(torch, "cpu", [3.5], [12.0]) == ([3.5], [12.0])
