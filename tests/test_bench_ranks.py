"""The bench's multi-rank logic on CPU ranks (gloo, world size 2).

One process per GPU runs its own replica of the block step: the job's step time is the
slowest rank's (one all-reduce of the per-rank times) and its rate counts every rank's
tokens.  The reference arm runs on rank 0 alone; the other ranks leave without work."""
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


def _rank_main(rank, world, port, local_ms, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.job_rate(local_ms[rank], 16384.0, world, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_counts_every_rank():
    world, local_ms = 2, [2.25, 3.5]  # rank 1 is the slower one
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), local_ms, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(world):
        ms, rate = res[r]
        assert ms == 3.5                                   # every rank reports the slowest
        assert rate == pytest.approx(world * 16384.0 / 3.5e-3)


def test_job_rate_on_one_rank():
    ms, rate = bench.job_rate(2.0, 16384.0, 1, "cpu")
    assert ms == 2.0
    assert rate == pytest.approx(16384.0 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 0

    bench.run_reference(Args(), 1, 2)  # rank 1 of 2: returns at once and prints nothing
    assert capsys.readouterr().out == ""
