"""The benchmark's multi-GPU path is replicas only: every rank runs the same
workload and the job is reported at the slowest rank's time. Its host logic
(max over ranks of the timed totals, whole-job rate, rank 0 alone runs the CPU
reference arm) is checked here with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 10 + r ms on the prefill and 2 - r ms on the decode
        local = {"prefill": 10.0 + rank, "decode": 2.0 - rank}
        tot = bench.max_over_ranks(local, torch.device("cpu"))
        rate = bench.job_rate(4.0e12, 5, world, tot["prefill"])
        dist.barrier()
        out[rank] = (tot["prefill"], tot["decode"], rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        pre, dec, rate = out[r]
        assert pre == 11.0 and dec == 2.0          # element-wise max over ranks
        assert rate == pytest.approx(2 * 4.0e12 * 5 / 0.011)


def test_single_process_is_identity():
    assert bench.max_over_ranks({"a": 1.5}, torch.device("cpu")) == {"a": 1.5}
    assert bench.job_rate(1.0, 4, 1, 2000.0) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    class Args:
        gpus, steps, warmup = 2, 1, 0
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(Args(), bench.PREFILL["single_head_n128_d64"], None)
    assert capsys.readouterr().out == ""          # rank 1 exits without work or output
