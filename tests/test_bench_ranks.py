"""Host side of bench.py's multi-rank run, on CPU with the gloo backend (world
size 2): the timing reduction takes the slowest rank, the whole-job value counts
every rank's units, and the reference arm runs on rank 0 only."""
import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        m = bench.max_over_ranks(times[rank], world)
        out[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world, times = 2, [12.5, 40.25]
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert dict(out) == {0: 40.25, 1: 40.25}


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    raw = 536870912  # one llama8b step of input
    one = bench.job_throughput(raw, 1, 100, 68.0)
    two = bench.job_throughput(raw, 2, 100, 68.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(raw * 100 / 0.068 / 1e9)
    # a slower rank lowers the whole job's value
    assert bench.job_throughput(raw, 2, 100, 80.0) < two


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, warmup, steps, reference_steps, oracle_layers, oracle_seconds = "tiny", 3, 1, 1, 0, 1.0

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args())
    assert buf.getvalue() == ""
