"""bench.py's own arm on CPU: the JSON line carries every key of the bench contract.

The GPU measurements are replaced by fixed stand-ins (this checks how the line is
assembled, not the numbers); the GPU run of the same code is the round's bench.
"""
import argparse
import json

import bench


class _FakeCtx:
    rank, ws = 0, 1

    def __init__(self):
        pass


def _fake_prefill(cx, args):
    roof = {"bound": "hbm", "achieved": 1.0, "peak": 2.0, "unit": "GB/s", "frac": 0.5, "traffic": None}
    return {"value": 1.25, "ms": 0.5, "tokens": 8192, "roofline": roof,
            "tensor": {"achieved": 1.0, "peak": 2.0, "unit": "TFLOP/s", "frac": 0.5},
            "e2e": {"value": 1.0, "unit": "Mtok/s", "h2d_bytes_per_step": 10, "d2h_bytes_per_step": 5},
            "launches": 8, "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
            "variants": {"plain_us": 500.0}, "chain_bound": {"us": 250.0, "frac": 0.5, "what": "chain"}}


def test_our_arm_json_line(monkeypatch, capsys):
    from linear_attention_chunkwise_gb300 import _build
    monkeypatch.setattr(_build, "build", lambda *a, **k: None)
    monkeypatch.setattr(bench, "Ctx", _FakeCtx)
    monkeypatch.setattr(bench, "bench_prefill", _fake_prefill)
    monkeypatch.setattr(bench, "bench_decode", lambda cx, args: {"value": 1.0})
    monkeypatch.setattr(bench, "bench_backward", lambda cx, args: {"value": 1.0})
    monkeypatch.setattr(bench, "bench_prefill_workload", lambda cx, args, name, calls: {"value": 1.0, "name": name})
    monkeypatch.setattr(bench, "cpu_baseline",
                        lambda s: {"value": 0.01, "unit": "Mtok/s", "cores": 16, "kind": "oracle", "sample": "x"})
    args = argparse.Namespace(steps=7, warmup=3, only="all", no_cpu_baseline=False, cpu_seconds=1.0)
    bench.run_ours(args)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["steps"] == 7 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert "workload" in d["config"] and "l2" in d["config"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in d["e2e"], key
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["gpu_launches"] > 0
    assert "decode" in d and "backward" in d
    assert set(d["prefill_workloads"]) == {"varlen_prefill", "long_prefill_1m"}
    assert d["chain_bound"]["us"] > 0 and 0 < d["chain_bound"]["frac"]
