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
