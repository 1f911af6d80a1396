"""The benchmark's multi-rank plumbing on CPU with the gloo backend (world size 2):
barrier, max-over-ranks step time, whole-job value, and the reference arm's
rank-0-only rule.  No GPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        ms = 1.0 + rank           # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, world)
        q.put((rank, ms_max, bench.job_value(world, 8192, ms_max)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, value in res:
        assert ms_max == 2.0                       # the slowest rank sets the step time
        assert value == pytest.approx(2 * 8192 / 0.002)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(1, 8192, 2.0) == pytest.approx(8192 / 0.002)
