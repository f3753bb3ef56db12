"""The multi-rank path of bench.py on CPU (gloo, world size 2): the layer
runs as independent replicas, one per GPU, so the only cross-rank steps are
the job's time (the maximum over ranks) and the whole-job rate (the units of
all ranks over that time).  Each rank here reports a different local time."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 25.0 * rank  # the second replica is slower
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        out[rank] = (ms, bench.job_rate(1000.0, 4, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_time_is_the_slowest_and_rate_counts_both():
    world = 2
    out = mp.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 125.0
    # 2 ranks x 1000 units x 4 steps in 0.125 s
    assert out[0][1] == pytest.approx(2 * 1000 * 4 / 0.125)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    assert bench.job_rate(10.0, 3, 1, 1000.0) == pytest.approx(30.0)
