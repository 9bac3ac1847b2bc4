"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the timed
region's max over ranks and the weak-scaling aggregate.  No GPU."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = 1.0 + rank * 0.5          # rank 1 is the slow one
        mx = bench.max_over_ranks(ms, world)
        flops = 1e12
        value = world * flops / (mx * 1e-3) / 1e12
        out[rank] = (mx, value)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(1.5) and res[1][0] == pytest.approx(1.5)
    # two replicas of 1 TFLOP each, slowest rank 1.5 ms
    assert res[0][1] == pytest.approx(2e12 / 1.5e-3 / 1e12)
