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


def _stub_arm(args):
    """The CUDA arm stood in for by its host logic on gloo: each rank reports
    the slowest rank's time and the whole-job value."""
    import torch
    import bench
    world, rank, local = bench.dist_env()
    bench.init_dist(world, "gloo")
    bench.barrier(world)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)
    value = bench.whole_job_value(1000, 4, world, slowest)
    with open(os.path.join(args.out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{rank} {local} {world} {slowest} {value}")
    torch.distributed.destroy_process_group()


def test_launcher_starts_one_rank_per_gpu(tmp_path, monkeypatch):
    # bench.py --gpus 2 without torchrun: bench starts the two ranks itself
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = bench.parse_args(["--gpus", "2"])
    args.out_dir = str(tmp_path)
    bench.launch_ranks(2, _stub_arm, args)
    got = sorted((tmp_path / f"rank{r}.txt").read_text().split() for r in range(2))
    for r, (rank, local, world, slowest, value) in enumerate(got):
        assert int(rank) == r and int(local) == r and int(world) == 2
        assert float(slowest) == 15.0
        assert float(value) == pytest.approx(2 * 1000 * 4 / 0.015)


def test_gpus_must_match_torchrun_world(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit, match="WORLD_SIZE=1"):
        bench.main(["--gpus", "2"])


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
