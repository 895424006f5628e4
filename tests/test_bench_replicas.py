"""The multi-process side of bench.py on CPU (gloo, world size 2): replicas
only, so the one collective is the job time, the longest rank's timed region,
which every rank must receive; the whole-job rate counts every rank's tokens
over that time.  The reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_elapsed(times[rank], world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_on_every_rank():
    world = 2
    times = [0.125, 0.5]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 0.5, 1: 0.5}
    # 8 query tokens per rank, 100 steps, over the job's 0.5 s
    assert bench.job_value(world, 8, 100, 0.5) == pytest.approx(3200.0)
    assert bench.job_elapsed(0.25, 1, "cpu") == 0.25


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys_argv = sys.argv
    try:
        sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
        args = bench.parse()
    finally:
        sys.argv = sys_argv
    assert bench.run_reference(args, 1, 2) == 0
    assert capsys.readouterr().out == ""
