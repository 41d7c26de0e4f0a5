"""The multi-rank path of bench.py on CPU: two gloo ranks.

Each rank runs its own batch (the attention partitions over (b, h) with no
exchange), so the only cross-rank operations are the barrier and the
max-over-ranks of the elapsed time; the whole-job value is the units every
rank processed over the slowest rank's time.
"""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import bench
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    elapsed = 10.0 + 5.0 * rank                 # rank 1 is the slow one
    slowest = bench.max_over_ranks(elapsed, world)
    value = bench.whole_job_value(1000, 4, world, slowest)
    q.put((rank, slowest, value))
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 1000 * 4 / 0.015)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.reference_arm(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert capsys.readouterr().out == ""


def test_single_rank_value():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_value(10, 2, 1, 1000.0) == 20.0
