"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

With N GPUs the benchmark runs N independent replicas (the decode path has
no exchange step): the job's step time is the slowest rank's, and the job
throughput counts the rows of every rank.  The reference arm runs on rank 0
only; other ranks return without work or output.
"""
import os
import socket

import pytest
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


def test_algorithmic_bytes_follow_the_record_sizes():
    """The metric's denominator: per (token, row, head, layer) the four loop calls
    of a shared-anchor group read 2 * (3 * (72 + 42) + 72) = 828 bytes at d = 128,
    g = 32 (anchor record 64 + 8, residual record 32 + 8 + 2, K and V); chained
    loop l reads the anchor and the residual planes of loops l .. P-2."""
    import synth
    w = synth.WORKLOADS["ouro8k"]
    B, N = w.batch, w.context
    rows = B * w.num_heads
    small = rows * (3 * 128 * 2 + 128 * 4)
    shared = bench.algorithmic_bytes_per_step(w, B, N)
    assert shared["per_loop"] == [2 * (72 + 42) * N * rows + small] * 3 + [2 * 72 * N * rows + small]
    append = rows * 2 * ((64 + 8) + 3 * (32 + 8 + 2)) + rows * 4 * 2 * 128 * 2
    assert shared["step"] == w.num_layers * (sum(shared["per_loop"]) + append)
    assert abs(shared["step"] - 10.42e9) / 10.42e9 < 0.01   # 828 B x 8192 x 64 x 24
    chained = bench.algorithmic_bytes_per_step(w, B, N, chained=True)
    assert chained["per_loop"][0] == 2 * (72 + 3 * 42) * N * rows + small
    assert chained["per_loop"][2] == shared["per_loop"][2]


def test_reference_arm_step_is_the_timed_sample(monkeypatch, capsys):
    """The reference arm's step is one bounded oracle sample: its ms_per_step is
    the sample's own time (steps x ms_per_step fits the run's clock), and its
    tokens/s counts the fraction of a decode step the samples covered."""
    import json
    import time
    import types

    import synth
    monkeypatch.setenv("RANK", "0")
    w = synth.WORKLOADS["toy"]
    args = types.SimpleNamespace(ref_budget=0.05, steps=3, warmup=1, gpus=1, chained=False)
    t0 = time.perf_counter()
    bench.run_reference(args, w)
    wall_ms = (time.perf_counter() - t0) * 1e3
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3
    assert 0 < line["ms_per_step"] * line["steps"] <= wall_ms
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
