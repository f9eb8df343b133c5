"""The multi-replica aggregation of bench.py on two gloo ranks (CPU): the job's step time is
the slowest rank's, and the throughput counts every rank's work."""
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
    ms = [10.0, 25.0][rank]
    value, ms_max = bench.aggregate_tflops(1e12, ms, world, device="cpu")
    out[rank] = (value, ms_max)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
    for r in range(world):
        value, ms_max = out[r]
        assert ms_max == pytest.approx(25.0)
        assert value == pytest.approx(2 * 1e12 / 25e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    value, ms = bench.aggregate_tflops(2e12, 4.0, 1, device="cpu")
    assert ms == 4.0 and value == pytest.approx(500.0)
    assert torch is not None
