"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

With N GPUs the benchmark runs N independent replicas (the decode path has
no exchange step): the job's step time is the slowest rank's, and the job
throughput counts the rows of every rank.  The reference arm runs on rank 0
only; other ranks return without work or output.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 7.5 * rank                       # rank 1 is the slow one
        slowest = bench.reduce_max_over_ranks(ms)
        value = bench.job_throughput(world, 4, slowest)
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{slowest} {value}\n")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput(tmp_path):
    world = 2
    tmp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    rows = [open(tmp_path / f"r{r}.txt").read().split() for r in range(world)]
    for slowest, value in rows:
        assert float(slowest) == 17.5                # every rank sees the slowest rank's time
        assert float(value) == pytest.approx(world * 4 / 17.5e-3)


def test_single_process_needs_no_group():
    assert not dist.is_initialized()
    assert bench.reduce_max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1, 4, 5.0) == pytest.approx(800.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(None, None)                  # returns before touching its arguments
    assert capsys.readouterr().out == ""
