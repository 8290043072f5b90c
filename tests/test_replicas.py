"""The multi-GPU bench runs independent replicas (nothing in the layer step is
exchanged between GPUs); its only cross-rank logic is the job rate: the slowest
rank's step time and the steps of all ranks over it.  Checked here with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms, value = bench.job_rate(1.0 + rank, world)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_job_rate_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    for r in range(world):
        ms, value = out[r]
        assert ms == pytest.approx(2.0)                 # the slowest rank's step time
        assert value == pytest.approx(world * 1000.0 / 2.0)


def test_job_rate_one_rank():
    import bench
    assert bench.job_rate(4.0, 1) == (4.0, 250.0)
