"""The replica (N>1) path of bench.py on CPU: two gloo ranks, each with its own
timing; the job's throughput counts every rank's rows over the slowest rank."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 100.0 if rank == 0 else 250.0
    value, ms_max = bench.aggregate(ms_local, rows_per_step=1000, steps=10, dist=dist, device="cpu")
    out[rank] = (value, ms_max)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, ms_max = res[r]
        assert ms_max == pytest.approx(250.0)
        assert value == pytest.approx(world * 1000 * 10 / 0.25)


def test_single_process_aggregate():
    import bench
    value, ms_max = bench.aggregate(50.0, rows_per_step=7, steps=4, dist=None, device="cpu")
    assert ms_max == 50.0 and value == pytest.approx(7 * 4 / 0.05)
