"""The multi-process path of bench.py on CPU: two gloo ranks (127.0.0.1)
run the same max-over-ranks reduction the benchmark applies to its CUDA-event
totals, and the whole-job throughput is computed from the slowest rank.
Decode and prefill shard by sequence with no exchange, so each GPU runs an
independent replica; the only cross-rank steps are the barrier and this
reduction.  The reference arm under torchrun runs on rank 0 alone."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = [12.5, 20.0][rank]  # rank 1 is the slow one
        dist.barrier()
        total = bench.max_over_ranks(local_ms, torch.device("cpu"), ws)
        value = bench.job_throughput(ws, 64, 10, total)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"total": total, "value": value}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank(tmp_path):
    ws = 2
    mp.spawn(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(ws)]
    for r in res:
        assert r["total"] == 20.0
        assert r["value"] == pytest.approx(2 * 64 * 10 / 0.020)


def test_single_rank_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(7.25, torch.device("cpu"), 1) == 7.25
    assert bench.job_throughput(1, 64, 50, 5000.0) == pytest.approx(640.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    class Args:
        steps, warmup = 2, 3
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""
