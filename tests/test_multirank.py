"""The N>1 path of bench.py on CPU: two gloo ranks, each with its own batch and
timings, no data-path collective; the reported time is the MAX over ranks and
the value counts every rank's bytes (weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks([1.0 + rank, 2.0 * (rank + 1), 0.5], dist)
    value = bench.weak_scaling_value(1_000_000, world, ms[0])
    out[rank] = ms + [value]
    dist.destroy_process_group()


def test_two_ranks_take_the_max_and_sum_the_work():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r][:3] == [2.0, 4.0, 0.5]
        assert out[r][3] == pytest.approx(2 * 1_000_000 / 2e-3 / 1e9)
