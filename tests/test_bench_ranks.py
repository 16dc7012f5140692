"""The benchmark's multi-rank host logic on CPU (gloo, two ranks): the step
shards into independent replicas, so the job's time is the slowest rank's
and its throughput counts every rank's bytes; the reference arm runs on
rank 0 alone."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        out[rank] = bench.job_time_ms(local_ms, dist, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == 5.0


def test_single_rank_time_is_local():
    assert bench.job_time_ms(4.5, None, None) == 4.5


def test_whole_job_throughput_counts_every_rank():
    one = bench.whole_job_tbs(1, 51e6, 18.0)
    assert one == pytest.approx(51e6 / 18e-6 / 1e12)
    assert bench.whole_job_tbs(4, 51e6, 18.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class A:  # the arguments run_reference reads
        config, steps, warmup, gpus = "tiny", 1, 0, 2
    bench.run_reference(A(), rank=1)
    assert capsys.readouterr().out == ""
