"""The bench's multi-rank aggregation on CPU (gloo, world size 2): every rank gets the slowest
rank's time, and the whole-job throughput is all ranks' tokens over that time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        max_ms = bench.slowest_rank_ms(times[rank], dist)
        out[rank] = (max_ms, bench.replica_throughput(world, 10, 15, max_ms))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_throughput_gloo_world2():
    world, port = 2, _free_port()
    times = [12.5, 20.0]   # ms: rank 1 is the slow one
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        max_ms, value = res[r]
        assert max_ms == 20.0
        assert value == pytest.approx(world * 10 * 15 / 0.020)


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(7.25) == 7.25
    assert bench.replica_throughput(1, 4, 15, 2.0) == pytest.approx(4 * 15 / 0.002)
