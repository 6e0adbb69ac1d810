"""The multi-GPU path of the benchmark runs independent replicas (the layer has
no cross-device exchange).  Its host-side aggregation - the barrier, the max of
the ranks' times and the whole-job throughput - runs here with two gloo ranks
on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(True)
        local_ms = 10.0 * (rank + 1)                  # rank 1 is the slowest
        value, slowest = bench.replica_throughput(1000, local_ms, world, True, torch.device("cpu"))
        out[rank] = (value, slowest)
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas_aggregate_like_the_benchmark():
    world = 2
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        value, slowest = res[rank]
        assert slowest == pytest.approx(20.0)                    # max over ranks, on every rank
        assert value == pytest.approx(world * 1000 / 0.020)      # all ranks' units / slowest time


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    value, slowest = bench.replica_throughput(500, 5.0, 1, False, torch.device("cpu"))
    assert slowest == 5.0 and value == pytest.approx(500 / 0.005)
