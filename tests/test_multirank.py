"""The benchmark's multi-rank bookkeeping on CPU, with world-size-2 gloo
process groups: every per-phase time of the job is the slowest rank's, the
whole-job throughput counts the work of all ranks over that time, and only
rank 0 runs and prints the CPU reference arm.  The layer itself needs no
exchange between ranks (output columns are independent), so this is the
whole of the multi-GPU path."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)]
        out[rank] = bench.max_over_ranks(mine, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_times_are_the_slowest_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()      # no fork of this (multi-threaded) process
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    expect = [2.0, 10.0, 10.0]
    assert out[0] == expect and out[1] == expect


def test_single_process_is_the_identity():
    assert bench.max_over_ranks([3.5, 1.25], torch.device("cpu")) == [3.5, 1.25]


def test_job_throughput_counts_every_rank():
    # two ranks each moving 122 MB per step, 10 steps, slowest rank 2.5 ms
    one = bench.job_gbs(122e6, 10, 2.5, 1)
    assert one == pytest.approx(122e6 * 10 / 2.5e-3 / 1e9)
    assert bench.job_gbs(122e6, 10, 2.5, 2) == pytest.approx(2 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    def no_oracle():
        raise AssertionError("rank 1 must not touch the oracle")

    monkeypatch.setattr(bench, "_oracle_setup", no_oracle)
    args = type("A", (), {"steps": 1, "warmup": 3})()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
