"""Host logic of bench.py's N > 1 path on CPU: two gloo ranks (spawned
processes, 127.0.0.1) agree on the slowest rank's time and on the whole-job
throughput; the oracle arm runs on rank 0 only. The GPU path uses the same
functions over NCCL."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        b.rank_barrier(world)
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        max_ms = b.max_over_ranks(local_ms, world, "cpu")
        value = b.job_throughput(max_ms / 1e3, world, 4096 * 10)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
            json.dump({"local_ms": local_ms, "max_ms": max_ms, "value": value}, fh)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["max_ms"] == 15.0  # the slowest rank's time, on every rank
        # every rank's 40,960 tokens over 15 ms
        assert r["value"] == pytest.approx(2 * 40960 / 0.015, rel=1e-12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.job_throughput(0.5, 1, 1000) == 2000.0
    bench.rank_barrier(1)  # no-op


def test_oracle_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1",
                                      "--warmup", "1"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""  # rank 1 prints nothing and does no work
