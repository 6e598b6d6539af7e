"""The multi-GPU path of bench.py is replicas: every rank runs the whole
layer set on its own GPU, with no collective on the data path.  The host
logic that turns per-rank times into the job's line -- the max over ranks
and the whole-job throughput -- is checked here with two gloo ranks on CPU."""

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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = [2.0, 3.0][rank]  # the second replica is the slower one
        out[rank] = (bench.max_over_ranks(dist, ms), bench.whole_job(dist, world, 1.5e9, ms),
                     bench.max_over_ranks(dist, float(rank)))
    finally:
        dist.destroy_process_group()


def test_replicas_two_gloo_ranks():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        mx, value, rmax = res[r]
        assert mx == 3.0  # every rank sees the slowest replica's time
        assert value == pytest.approx(world * 1.5e9 / 3.0 / 1e6)  # all ranks' bytes over that time
        assert rmax == 1.0


def test_single_rank_needs_no_group():
    import bench

    assert bench.max_over_ranks(None, 4.0) == 4.0
    assert bench.whole_job(None, 1, 2e9, 2.0) == pytest.approx(1000.0)
    assert torch.__version__
