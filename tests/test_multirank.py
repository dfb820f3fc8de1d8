"""Host logic of the N-process benchmark on CPU: world_size-2 `gloo` ranks.

The layer forward does not shard: under torchrun every rank runs an
independent replica on its own GPU, and the job's throughput is the units
all ranks processed over the slowest rank's time.  These tests run that
bookkeeping (process-group setup, max over ranks, the job rate, teardown) in
two CPU processes, and check that the reference arm's non-zero ranks exit
without work."""
from __future__ import annotations

import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str, local_s: list):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench

    w, r, local = bench.dist_setup()
    dev = torch.device("cpu")
    bench.barrier(w)
    slowest = bench.max_over_ranks(local_s[r], w, dev)
    rate, t = bench.job_rate(1000.0, local_s[r], w, dev)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "slowest": slowest, "rate": rate, "t": t}, f)
    bench.dist_teardown(w)


def test_two_gloo_ranks_agree_on_the_slowest_rank(tmp_path):
    world = 2
    local_s = [0.5, 2.0]  # rank 1 is the slow replica
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path), local_s), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert (d["world"], d["rank"], d["local"]) == (world, r, r)
        assert d["slowest"] == 2.0 and d["t"] == 2.0
        # 2 ranks x 1000 units over the slowest rank's 2 s
        assert d["rate"] == pytest.approx(1000.0)


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.job_rate(300.0, 1.5, 1, torch.device("cpu")) == (200.0, 1.5)
    bench.barrier(1)
    bench.dist_teardown(1)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    def boom(*a, **k):
        raise AssertionError("rank 1 of the reference arm must not build the workload")

    monkeypatch.setattr(bench.synth, "make_activations", boom)
    args = type("A", (), {"gpus": 2, "steps": 1, "warmup": 3})()
    bench.run_reference(args)
    assert capsys.readouterr().out == ""
    import torch.distributed as dist
    assert not dist.is_initialized()
