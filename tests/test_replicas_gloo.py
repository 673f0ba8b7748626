"""bench.py's N-replica timing over world_size-2 gloo ranks on the CPU: the step
time is the maximum over ranks and the throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    def rank_max(x):
        t = torch.tensor([x], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    local_ms = 100.0 + 25.0 * rank            # rank 1 is the slow one
    ms, rate = bench.aggregate_over_ranks(local_ms, 32768, world, rank_max)
    out[rank] = (ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_max_over_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == pytest.approx(125.0)
        assert rate == pytest.approx(2 * 32768 / 0.125)


def test_single_rank_is_identity():
    import bench
    ms, rate = bench.aggregate_over_ranks(50.0, 1000, 1, None)
    assert ms == 50.0 and rate == pytest.approx(20000.0)
