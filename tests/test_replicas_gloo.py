"""Multi-GPU bench path, host side: replicas (no data-path collective), whole-job
throughput = all ranks' tokens over the slowest rank's time. Two gloo ranks on
the CPU run the same reduction code bench.py runs under torchrun."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    secs = [0.5, 0.8][rank]                      # rank 1 is the slow one
    tokens = 1000.0
    slowest = bench.max_over_ranks(secs, world, device="cpu")
    total = bench.sum_over_ranks(tokens, world, device="cpu")
    bench.barrier(world)
    results[rank] = (slowest, total, total / slowest)
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_the_slowest_rank():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    old = os.environ.get("PYTHONPATH", "")
    os.environ["PYTHONPATH"] = root + (os.pathsep + old if old else "")
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, results), nprocs=2, join=True, start_method="spawn")
    assert set(results.keys()) == {0, 1}
    for r in (0, 1):
        slowest, total, value = results[r]
        assert slowest == 0.8 and total == 2000.0
        assert value == pytest.approx(2500.0)


def test_aggregate_formula():
    import bench
    assert bench.aggregate([10, 10, 10], [1.0, 2.0, 0.5]) == 15.0
