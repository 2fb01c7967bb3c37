"""The multi-rank host path of bench.py on the CPU: two gloo ranks.

On GPUs the ranks are independent replicas (no data-path collective); what
the ranks share is the timing protocol (barrier, then the slowest rank's
time) and the whole-job throughput, and the reference arm runs on rank 0
alone. These run here with the gloo backend, world size 2, on 127.0.0.1.
"""
import argparse
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = ms
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_time():
    world, port = 2, _free_port()
    times = [3.5, 5.25]
    out = mp.get_context("spawn").Manager().list([0.0, 0.0])
    mp.start_processes(_rank_main, args=(world, port, times, out), nprocs=world,
                       start_method="spawn", join=True)
    assert list(out) == [5.25, 5.25]


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.0, 1) == 4.0


def test_job_throughput_counts_every_rank_over_the_slowest_time():
    # 2 replicas of 3.849 TFLOP each, slowest rank 5 ms: 1539.6 TFLOP/s
    assert bench.job_tflops(3.849e12, 2, 5.0) == pytest.approx(1539.6)
    assert bench.job_tflops(3.849e12, 1, 5.0) == pytest.approx(769.8)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # under torchrun, ranks other than 0 exit at once without work or output
    monkeypatch.setenv("RANK", "1")
    ns = argparse.Namespace(workload="usp_ud2_ring4_s8k", seed=0, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(ns) is None
    assert capsys.readouterr().out == ""
