"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

Each rank runs its own independent problem (no collective on the data path);
the only collective is the max of the per-rank step time, and rank 0 reports
tokens of all ranks / slowest rank.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        local_ms = 1.0 + rank  # the slower rank decides the step time
        ms = bench.max_over_ranks(dist, local_ms, "cpu")
        out[rank] = (ms, bench.whole_job_mtok_s(8192, world, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == pytest.approx(2.0) and res[1][0] == pytest.approx(2.0)
    assert res[0][1] == pytest.approx(8192 * 2 / 2e-3 / 1e6)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(dist, 3.5, "cpu") == 3.5
    assert bench.whole_job_mtok_s(8192, 1, 1.0) == pytest.approx(8.192)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.argparse.Namespace(steps=1, warmup=0, cpu_seconds=1.0))
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line(monkeypatch, capsys):
    """Rank 0 prints one JSON line with the contract's keys, the oracle as the reference."""
    import json
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    bench.run_reference(bench.argparse.Namespace(steps=1, warmup=0, cpu_seconds=0.5))
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] == d["e2e"]["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
