"""The bench's multi-GPU form on CPU: world_size-2 process groups over gloo.

The path does not shard (replicas only): every rank scores its own copy of
the workload, the timed regions are combined by one all-reduce of their
maxima, and rank 0 alone reports the whole job's rate, N times the tokens of
one replica over the slowest rank's time. The reference arm runs on rank 0
only; the other ranks return without work.
"""

import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 10 + r ms for the headline region and 30 - r for e2e
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world, torch.device("cpu"))
        results[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    # every rank sees the element-wise maximum of the two ranks' timings
    assert results[0] == [11.0, 30.0] and results[1] == [11.0, 30.0]


def test_single_rank_keeps_its_own_timing():
    import torch
    assert bench.max_over_ranks([3.5, float("inf")], 1, torch.device("cpu")) == [3.5, float("inf")]


def test_whole_job_rate_counts_every_replica():
    # two replicas of 32768 tokens, 10 steps, the slowest rank's region 2 ms
    assert bench.whole_job_rate(2, 32768, 10, 2.0) == pytest.approx(2 * 32768 * 10 / 2e-3)
    assert bench.whole_job_rate(1, 32768, 10, 2.0) == pytest.approx(32768 * 10 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    args = bench.parse(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args, rank=1, world=2)   # returns before any work
    assert capsys.readouterr().out == ""


def test_rank_and_world_come_from_the_launcher_environment(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_info() == (1, 4, 1)
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v)
    assert bench.dist_info() == (0, 1, 0)
