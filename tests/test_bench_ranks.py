"""bench.py's multi-rank (replica) aggregation on CPU with the gloo backend.

Each rank times its own full product; ranks agree on the slowest rank's time
and report whole-job throughput = world x FLOP / that time.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = 2.0 + rank  # rank 1 is the slow one
    ms, value = bench.combine_ranks(ms_local, 137.438953472e9, world)
    results[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn",
                           join=True)
        res = dict(results)
    assert set(res) == {0, 1}
    for ms, value in res.values():
        assert ms == 3.0
        assert abs(value - 2 * 137.438953472e9 / 3.0e-3 / 1e12) < 1e-9


def test_single_rank_needs_no_process_group():
    import bench
    ms, value = bench.combine_ranks(2.5, 1e12, 1)
    assert ms == 2.5 and abs(value - 1e12 / 2.5e-3 / 1e12) < 1e-12
