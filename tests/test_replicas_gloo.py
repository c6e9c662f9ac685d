"""The multi-GPU path of bench.py is replicas only (requests and heads are
independent; the path has no exchange step).  Its host logic -- the
max-over-ranks time and the whole-job value -- is checked here with two gloo
ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world, device="cpu")
        out[rank] = slowest
        out[2 + rank] = bench.whole_job_value(1e12, slowest, world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_on_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().list([0.0] * 4)
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
    assert list(out[:2]) == [20.0, 20.0]
    # 2 replicas x 1e12 FLOP in 20 ms -> 100 TFLOP/s for the whole job
    assert out[2] == pytest.approx(100.0) and out[3] == pytest.approx(100.0)


def test_single_rank_is_a_no_op():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.0, 1) == 7.0
    assert bench.whole_job_value(2e12, 10.0, 1) == pytest.approx(200.0)
