#!/usr/bin/env python
"""Benchmark of the KDA hot path on GB300: chunkwise prefill + fused decode.

One step = one kda_prefill call on the 8k workload (B=1, H=32, T=8192,
d=128, bf16 q/k/v, fp32 gates, fp32 state, S0 = 0).  `value` is prefill
throughput in Mtok/s (sequence positions, all 32 heads) with inputs resident
in HBM; the inputs (404 MB per step) are larger than L2, so no flush is
needed between steps.  The same JSON line carries the decode workload
(256 sequences x 32 heads, 100 consecutive steps in one CUDA graph) as
state GB/s under "decode".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same per-GPU workload on its own GPU (the
(sequence, head) units are independent: weak scaling, no collective on the
data path); the step time is the max over ranks.  `--impl reference` times
the fp64 CPU oracle on the host cores instead (bounded token samples).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

PREFILL_WORKLOAD = "prefill_8k"
DECODE_WORKLOAD = "decode_256x32"
H, D = 32, 128
# algorithmic bytes / flops per token-head (q, k, v bf16 + log_alpha fp32 + beta fp32 + o bf16)
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * D * 2 + D * 4 + 4 + D * 2          # 1540
PREFILL_FLOPS_PER_TOKEN_HEAD = 10 * 64 * D + 6 * D * D                  # 180,224 (full 64x64 tiles)
STATE_BYTES = D * D * 4                                                 # 65,536
# backward: reads q, k, v, grad_o (bf16), log_alpha, beta; writes fp32 grad_q, grad_k, grad_v,
# grad_log_alpha and grad_beta
BACKWARD_BYTES_PER_TOKEN_HEAD = 4 * D * 2 + D * 4 + 4 + 4 * D * 4 + 4   # 3,592
# tensor-core work of the chunkwise backward per (chunk, head), multiply-adds: prep 3.67M (Grams,
# Qh^T dO, Tb^T Kb, Mm^T dO, Tb^T MdO), adjoint scan 2.10M, value 5.24M, key 6.29M
BACKWARD_MACS_PER_CHUNK_HEAD = (2 * 64 * 64 * 128 + 128 * 128 * 64 + 3 * 64 * 128 * 64
                                + 2 * 64 * 128 * 128
                                + 2 * 64 * 64 * 128 + 2 * 64 * 128 * 128 + 4 * 64 * 128 * 64
                                + 2 * 64 * 64 * 128 + 3 * 64 * 128 * 128 + 4 * 64 * 128 * 64)
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rate
DECODE_BYTES_PER_UNIT = 2 * STATE_BYTES + PREFILL_BYTES_PER_TOKEN_HEAD  # 132,612
METRIC = "KDA prefill Mtok/s & % tensor peak; decode state GB/s & % HBM (H=32, d=128)"
# sources whose ncu DRAM counters profiles/ncu_traffic.json records (null once they change)
PREFILL_SOURCES = ["kda_api.cu", "kda_prefill_split.cu", "kda_prefill_common.cuh", "kda_ptx.cuh", "kda_internal.h"]
DECODE_SOURCES = ["kda_decode.cu", "kda_ptx.cuh", "kda_internal.h"]
BACKWARD_SOURCES = ["kda_api.cu", "kda_backward.cu", "kda_prefill_split.cu", "kda_prefill_common.cuh", "kda_ptx.cuh",
                    "kda_internal.h"]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return dict(hbm=float(pk["hbm_gbs"]), bf16=float(pk["bf16_tflops"]),
                    bf16_sustained=float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "linear_attention_chunkwise_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, src_files):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            rec = json.load(fh)[kernel]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(src_files):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """SM clocks, power and clock-event (throttle) reasons sampled DURING a timed
    region: NVML through ctypes every ~2 ms (short regions still get samples),
    falling back to `nvidia-smi -lms 200`.  Read-only: no setting is changed."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.samples = []      # (sm_mhz, max_mhz, reasons_mask, power_w)
        self._stop = threading.Event()
        self._t = None
        self._nvml = None
        self._handle = None
        self._smi = None

    def _init_nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        props = torch.cuda.get_device_properties(self.dev)
        bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
            raise RuntimeError("nvml handle")
        self._nvml, self._handle = lib, h
        fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self._reasons_fn = fn

    def _poll_nvml(self):
        import ctypes
        lib, h = self._nvml, self._handle
        clk, mx, pw = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            ok = lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self._reasons_fn(h, ctypes.byref(rs))
            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            if ok:
                self.samples.append((float(clk.value), float(mx.value), int(rs.value), pw.value / 1000.0))
            time.sleep(0.002)

    def _poll_smi(self):
        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,power.draw")
        self._smi = subprocess.Popen(["nvidia-smi", f"--query-gpu={fields}", "--format=csv,noheader,nounits",
                                      "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        bits = [0x8, 0x40, 0x20, 0x4]
        for line in self._smi.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                mask = sum(b for b, v in zip(bits, parts[2:6]) if v.lower() == "active")
                self.samples.append((float(parts[0]), float(parts[1]), mask, float(parts[6])))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        try:
            self._init_nvml()
            target = self._poll_nvml
            self.source = "nvml"
        except Exception:
            target = self._poll_smi
            self.source = "nvidia-smi"
        self._t = threading.Thread(target=target, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._smi is not None:
            self._smi.terminate()
        if self._t is not None:
            self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [x[0] for x in self.samples]
        mask = 0
        for x in self.samples:
            mask |= x[2]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(x[1] for x in self.samples),
                "reasons": sorted(v for b, v in self.REASONS.items() if mask & b),
                "power_w_max": round(max(x[3] for x in self.samples), 1),
                "samples": len(sm), "source": self.source}


# ------------------------------------------------------ multi-rank math ----

def max_over_ranks(dist, x: float, device) -> float:
    """Max of a per-rank scalar over all ranks (the step time every rank reports)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_mtok_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes its own problem; value = all tokens / slowest rank."""
    return tokens_per_rank * world / (ms_max * 1e-3) / 1e6


# ----------------------------------------------------------------- ours ----

class Ctx:
    """Process/device context shared by the two measurements."""

    def __init__(self):
        import torch
        import torch.distributed as dist
        self.torch, self.dist = torch, dist
        self.ws, self.rank, local = dist_env()
        if self.ws > 1:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            torch.cuda.set_device(0)
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stream = torch.cuda.current_stream()
        self.peaks = load_peaks()

    def barrier(self):
        if self.ws > 1:
            self.dist.barrier()
        self.torch.cuda.synchronize()

    def max_over_ranks(self, x: float) -> float:
        return max_over_ranks(self.dist, x, self.dev)

    def events(self):
        E = self.torch.cuda.Event
        return E(enable_timing=True), E(enable_timing=True)


class CopyOverlap:
    """End-to-end steps with the host<->device copies overlapped across steps.  Every step copies
    all of its inputs from pinned host memory to the device and reads its result back; step i+1's
    inputs travel (own stream) while step i computes, and step i's result travels back (own stream)
    while step i+1 computes.  Two device buffer sets, reused under events."""

    def __init__(self, torch, compute_stream, host_in, dev_in_sets, host_out, dev_out_sets):
        self.torch, self.cs = torch, compute_stream
        self.h2d, self.d2h = torch.cuda.Stream(), torch.cuda.Stream()
        self.host_in, self.dev_in = host_in, dev_in_sets
        self.host_out, self.dev_out = host_out, dev_out_sets
        E = torch.cuda.Event
        self.in_ready, self.in_free = [E(), E()], [E(), E()]
        self.out_ready, self.out_free = [E(), E()], [E(), E()]
        self.i = 0

    def start(self):  # copies issued from now on begin after everything already on the compute stream
        self.h2d.wait_stream(self.cs)
        self.d2h.wait_stream(self.cs)

    def step(self, compute):
        t, b = self.torch, self.i & 1
        self.h2d.wait_event(self.in_free[b])  # step i-2 no longer reads this input set
        with t.cuda.stream(self.h2d):
            for d, h in zip(self.dev_in[b], self.host_in):
                d.copy_(h, non_blocking=True)
        self.in_ready[b].record(self.h2d)
        self.cs.wait_event(self.in_ready[b])
        self.cs.wait_event(self.out_free[b])  # step i-2's result has been read back
        compute(self.dev_in[b], self.dev_out[b])
        self.in_free[b].record(self.cs)
        self.out_ready[b].record(self.cs)
        self.d2h.wait_event(self.out_ready[b])
        with t.cuda.stream(self.d2h):
            for h, d in zip(self.host_out, self.dev_out[b]):
                h.copy_(d, non_blocking=True)
        self.out_free[b].record(self.d2h)
        self.i += 1

    def finish(self):  # the compute stream waits for the last copies
        self.cs.wait_stream(self.h2d)
        self.cs.wait_stream(self.d2h)


def piecewise_launches(seq_chunks: int, min_piece: int = 48, max_pieces: int = 32, lag: float = 0.05):
    """(pass-1 launches, scan launches) of the library's piecewise prefill schedule for one sequence
    of seq_chunks chunks: the piece count from pieces of max(min_piece, ceil(n / max_pieces)) chunks,
    then equal pieces of sq chunks; pass 1 a lead of sq + lag * sq * (pieces - 1) chunks, then
    equal shares."""
    sq0 = max(min_piece, -(-seq_chunks // max_pieces))
    n0 = -(-seq_chunks // sq0)
    sq = -(-seq_chunks // n0)
    pieces = -(-seq_chunks // sq)
    if pieces <= 1:
        return 1, 1
    lead = min(seq_chunks, sq + int(lag * sq * (pieces - 1) + 0.999))
    share = (seq_chunks - lead + pieces - 2) // (pieces - 1)
    prepared, n_prep = 0, 0
    for j in range(pieces):
        scan_end = min(seq_chunks, (j + 1) * sq)
        prep_end = max(lead if j == 0 else min(seq_chunks, lead + j * share), scan_end)
        if prep_end > prepared:
            n_prep += 1
            prepared = prep_end
    return n_prep, pieces


def bench_prefill(cx: Ctx, args):
    """Prefill on the 8k workload: device-resident timing, then end to end from pinned host memory."""
    torch = cx.torch
    import linear_attention_chunkwise_gb300 as kda
    from linear_attention_chunkwise_gb300 import synth

    c = synth.WORKLOADS[PREFILL_WORKLOAD]
    p = synth.prefill_inputs(c["lengths"], c["H"], D, c["dtype"], c["lo"], c["s0_std"],
                             synth.workload_seed(PREFILL_WORKLOAD) + 1000 * cx.rank, cx.dev)
    T = p.total_tokens
    o = torch.empty_like(p.q)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device=cx.dev)
    wsb = kda.kda_prefill_workspace_bytes(torch.bfloat16, 1, T, H)
    work = torch.empty(max(wsb, 256), dtype=torch.uint8, device=cx.dev)

    def step():
        kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, o=o, S_final=sf,
                        workspace=work, stream=cx.stream)

    for _ in range(args.warmup):
        step()
    cx.barrier()
    ev0, ev1 = cx.events()
    # clocks are sampled from the timed steps through the end-to-end, variant and chain timings below
    # (the same kernels), so that a short timed region still gets many samples
    clk = ClockSampler(cx.dev)
    clk.__enter__()
    ev0.record(cx.stream)
    for _ in range(args.steps):
        step()
    ev1.record(cx.stream)
    cx.barrier()
    ms_local = ev0.elapsed_time(ev1) / args.steps
    ms = cx.max_over_ranks(ms_local)
    tokens_per_step = T * cx.ws
    bytes_per_launch = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + H * STATE_BYTES  # + S_final write
    flops_per_launch = T * H * PREFILL_FLOPS_PER_TOKEN_HEAD
    achieved_gbs = bytes_per_launch / (ms_local * 1e-3) / 1e9
    achieved_tf = flops_per_launch / (ms_local * 1e-3) / 1e12

    # end to end through the same C-ABI call: pinned host inputs in, o and S_final out, every step;
    # the copies of neighbouring steps overlap this step's compute (CopyOverlap)
    names = ("q", "k", "v", "log_alpha", "beta", "cu_seqlens")
    host_in = [getattr(p, n).cpu().pin_memory() for n in names]
    dev_in = [[torch.empty_like(getattr(p, n)) for n in names] for _ in range(2)]
    o_host = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    sf_host = torch.empty(sf.shape, dtype=sf.dtype).pin_memory()
    dev_out = [[torch.empty_like(o), torch.empty_like(sf)] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = o_host.numel() * o_host.element_size() + sf_host.numel() * sf_host.element_size()
    pipe = CopyOverlap(torch, cx.stream, host_in, dev_in, [o_host, sf_host], dev_out)

    def e2e_compute(x, y):
        kda.kda_prefill(x[0], x[1], x[2], x[3], x[4], x[5], None, o=y[0], S_final=y[1], workspace=work,
                        stream=cx.stream)

    pipe.start()
    for _ in range(max(3, args.warmup)):
        pipe.step(e2e_compute)
    pipe.finish()
    cx.barrier()
    ev0.record(cx.stream)
    pipe.start()
    for _ in range(args.steps):
        pipe.step(e2e_compute)
    pipe.finish()
    ev1.record(cx.stream)
    cx.barrier()
    e2e_ms = cx.max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    del dev_in, dev_out

    # the same call with the fused prologue / epilogue, and with a state snapshot every 1024 tokens
    g = torch.Generator(device=cx.dev).manual_seed(7 + cx.rank)
    gate = torch.randn(p.q.shape, generator=g, device=cx.dev).to(p.q.dtype)
    wrms = torch.ones(D, dtype=torch.float32, device=cx.dev)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, out_gate=gate, rms_weight=wrms)
    snap_pos = torch.arange(1024, T + 1, 1024, dtype=torch.int32, device=cx.dev)
    snap_seq = torch.zeros_like(snap_pos)
    ss = torch.empty((snap_pos.numel(), H, D, D), dtype=torch.float32, device=cx.dev)

    def variant_us(fn, n=10):
        for _ in range(3):
            fn()
        cx.barrier()
        ev0.record(cx.stream)
        for _ in range(n):
            fn()
        ev1.record(cx.stream)
        cx.barrier()
        return round(cx.max_over_ranks(ev0.elapsed_time(ev1) / n) * 1e3, 1)

    variants = {
        "plain_us": round(ms * 1e3, 1),
        "fused_prologue_epilogue_us": variant_us(lambda: kda.kda_prefill_ex(
            p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, fusion=fz, o=o, S_final=sf, workspace=work,
            stream=cx.stream)),
        "fused_prologue_only_us": variant_us(lambda: kda.kda_prefill_ex(
            p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, fusion=kda.Fusion(l2norm_qk=True, beta_sigmoid=True),
            o=o, S_final=sf, workspace=work, stream=cx.stream)),
        "fused_epilogue_only_us": variant_us(lambda: kda.kda_prefill_ex(
            p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, fusion=kda.Fusion(out_gate=gate, rms_weight=wrms),
            o=o, S_final=sf, workspace=work, stream=cx.stream)),
        "snapshots_every_1024_us": variant_us(lambda: kda.kda_prefill_snapshots(
            p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, snap_seq, snap_pos, None, o=o, S_final=sf,
            S_snap=ss, workspace=work, stream=cx.stream)),
    }
    del gate, ss
    # the limit that binds this workload: the scan's serial chain over the sequence's 128 chunks.  The
    # same sequence with one head runs that chain with the GPU otherwise idle (pass 1 and the other heads'
    # chains are what the 32-head call adds); its time is the chain's floor for this sequence.
    p1 = synth.prefill_inputs(c["lengths"], 1, D, c["dtype"], c["lo"], c["s0_std"],
                              synth.workload_seed(PREFILL_WORKLOAD) + 1000 * cx.rank + 1, cx.dev)
    o1 = torch.empty_like(p1.q)
    sf1 = torch.empty((1, 1, D, D), dtype=torch.float32, device=cx.dev)
    chain_us = variant_us(lambda: kda.kda_prefill(p1.q, p1.k, p1.v, p1.log_alpha, p1.beta, p1.cu_seqlens, None,
                                                  o=o1, S_final=sf1, stream=cx.stream), n=20)
    del p1, o1, sf1
    clk.__exit__(None, None, None)
    chain = {"us": chain_us, "frac": round(chain_us / (ms * 1e3), 4),
             "what": "the same 8192-token sequence with 1 head: the scan's 128-chunk serial chain with the GPU "
                     "otherwise idle; frac = that floor / this call's time"}
    # kernels per call: the chunk table (one sequence: no schedule kernel) + the pass-1 and scan launches
    # of the piecewise schedule (the scan leaves SMs idle), else one prep + one scan
    sms = torch.cuda.get_device_properties(cx.dev).multi_processor_count
    n_prep, n_scan = piecewise_launches(-(-T // 64)) if 2 * H * 2 <= sms else (1, 1)
    pk = cx.peaks
    return {
        "value": whole_job_mtok_s(T, cx.ws, ms),
        "ms": ms,
        "launches": (1 + n_prep + n_scan) * args.steps,
        "variants": variants,
        "chain_bound": chain,
        "tokens": T,
        "roofline": {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved_gbs / pk["hbm"], 4),
                     "traffic": ncu_traffic("kda_prefill_two_pass", PREFILL_SOURCES),
                     "kernel": "kda_prefill call (chunk table + chunk prep + scan kernels)",
                     "peak_source": pk["src"] + " burst copy",
                     "bytes_per_launch": bytes_per_launch},
        "tensor": {"achieved": round(achieved_tf, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                   "frac": round(achieved_tf / pk["bf16"], 4), "flops_per_launch": flops_per_launch,
                   "peak_source": pk["src"] + " bf16 burst"},
        "e2e": {"value": round(tokens_per_step / (e2e_ms * 1e-3) / 1e6, 3), "unit": "Mtok/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "overlap": "H2D of step i+1 and D2H of step i-1 run beside step i (two buffer sets, "
                           "copy streams ordered by events)"},
        "clocks": dict(clk.summary(), window="the timed steps, then the end-to-end, variant and chain timings"),
    }


def bench_decode(cx: Ctx, args):
    """Decode: 256 x 32 heads, 100 consecutive steps captured in one CUDA graph."""
    torch = cx.torch
    import linear_attention_chunkwise_gb300 as kda
    from linear_attention_chunkwise_gb300 import synth

    dc = synth.WORKLOADS[DECODE_WORKLOAD]
    d = synth.decode_inputs(dc["N"], dc["H"], dc["steps"], D, dc["dtype"], dc["lo"], dc["s_std"],
                            synth.workload_seed(DECODE_WORKLOAD) + 1000 * cx.rank, cx.dev)
    n_units = dc["N"] * dc["H"]
    steps = dc["steps"]
    od = torch.empty((steps, dc["N"], dc["H"], D), dtype=torch.bfloat16, device=cx.dev)
    gstream = torch.cuda.Stream(device=cx.dev)
    kda.kda_decode_step(d.q[0], d.k[0], d.v[0], d.log_alpha[0], d.beta[0], d.S, None, o=od[0])  # load + warm
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gstream):
        for t in range(steps):
            kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], d.S, None, o=od[t])
    reps = max(1, args.decode_reps)
    for _ in range(max(1, args.warmup)):
        graph.replay()
    cx.barrier()
    ev0, ev1 = cx.events()
    # CUDAGraph.replay() launches on the current stream: time it there
    with ClockSampler(cx.dev) as clk:
        ev0.record(cx.stream)
        for _ in range(reps):
            graph.replay()
        ev1.record(cx.stream)
        cx.barrier()
    ms_local = ev0.elapsed_time(ev1) / (reps * steps)
    ms = cx.max_over_ranks(ms_local)
    state_gbs = cx.ws * n_units * 2 * STATE_BYTES / (ms * 1e-3) / 1e9
    achieved = n_units * DECODE_BYTES_PER_UNIT / (ms_local * 1e-3) / 1e9

    # multi-token step (speculative verify): T_MULTI tokens per sequence in one launch
    T_MULTI = 4
    dm = synth.decode_inputs(dc["N"], dc["H"], T_MULTI, D, dc["dtype"], dc["lo"], dc["s_std"],
                             synth.workload_seed(DECODE_WORKLOAD) + 5000 + 1000 * cx.rank, cx.dev)
    tm = lambda x: x.transpose(0, 1).contiguous()
    mq, mk, mv, mla, mb = tm(dm.q), tm(dm.k), tm(dm.v), tm(dm.log_alpha), tm(dm.beta)
    mo = torch.empty_like(mq)

    def multi_step():
        kda.kda_decode_multi(mq, mk, mv, mla, mb, dm.S, None, o=mo, stream=cx.stream)

    for _ in range(max(1, args.warmup)):
        multi_step()
    cx.barrier()
    n_multi = 50
    ev0.record(cx.stream)
    for _ in range(n_multi):
        multi_step()
    ev1.record(cx.stream)
    cx.barrier()
    m_ms = cx.max_over_ranks(ev0.elapsed_time(ev1) / n_multi)
    multi = {"tokens_per_launch_per_sequence": T_MULTI, "us_per_launch": round(m_ms * 1e3, 2),
             "tokens_per_s": round(cx.ws * n_units // dc["H"] * T_MULTI / (m_ms * 1e-3), 1),
             "state_gbs": round(cx.ws * n_units * 2 * STATE_BYTES / (m_ms * 1e-3) / 1e9, 1),
             "bytes_per_launch": n_units * (2 * STATE_BYTES + T_MULTI * PREFILL_BYTES_PER_TOKEN_HEAD),
             "hbm_frac": round(n_units * (2 * STATE_BYTES + T_MULTI * PREFILL_BYTES_PER_TOKEN_HEAD)
                               / (m_ms * 1e-3) / 1e9 / cx.peaks["hbm"], 4),
             "traffic": ncu_traffic("kda_decode_multi_kernel", DECODE_SOURCES)}
    del dm, mq, mk, mv, mla, mb, mo

    # decode step with the fused prologue / epilogue (L2 norm of q, k; sigmoid beta; RMSNorm x gate)
    gate = torch.randn(od[0].shape, device=cx.dev).to(od.dtype)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, out_gate=gate,
                    rms_weight=torch.ones(D, dtype=torch.float32, device=cx.dev))

    def fused_step():
        kda.kda_decode_step_ex(d.q[0], d.k[0], d.v[0], d.log_alpha[0], d.beta[0], d.S, None, fusion=fz, o=od[0],
                               stream=cx.stream)

    for _ in range(3):
        fused_step()
    cx.barrier()
    ev0.record(cx.stream)
    for _ in range(50):
        fused_step()
    ev1.record(cx.stream)
    cx.barrier()
    f_ms = cx.max_over_ranks(ev0.elapsed_time(ev1) / 50)
    fused = {"us_per_step": round(f_ms * 1e3, 2),
             "state_gbs": round(cx.ws * n_units * 2 * STATE_BYTES / (f_ms * 1e-3) / 1e9, 1)}
    del gate

    # end to end: each step's inputs H2D from pinned memory and its o D2H; the states stay in HBM;
    # the copies of neighbouring steps overlap this step's compute (CopyOverlap)
    names = ("q", "k", "v", "log_alpha", "beta")
    hq = [getattr(d, n)[0].cpu().pin_memory() for n in names]
    dq = [[getattr(d, n)[0].clone() for n in names] for _ in range(2)]
    oh = torch.empty(od[0].shape, dtype=od.dtype).pin_memory()
    dout = [[torch.empty_like(od[0])] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hq)
    d2h = oh.numel() * oh.element_size()
    pipe = CopyOverlap(torch, cx.stream, hq, dq, [oh], dout)

    def e2e_compute(x, y):
        kda.kda_decode_step(x[0], x[1], x[2], x[3], x[4], d.S, None, o=y[0], stream=cx.stream)

    pipe.start()
    for _ in range(3):
        pipe.step(e2e_compute)
    pipe.finish()
    cx.barrier()
    n_e2e = 100
    ev0.record(cx.stream)
    pipe.start()
    for _ in range(n_e2e):
        pipe.step(e2e_compute)
    pipe.finish()
    ev1.record(cx.stream)
    cx.barrier()
    e2e_ms = cx.max_over_ranks(ev0.elapsed_time(ev1) / n_e2e)
    pk = cx.peaks
    return {
        "workload": "KDA decode step, 256 sequences x 32 heads, d=128, bf16 q/k/v, fp32 states (512 MiB) "
                    "updated in place, 100 consecutive steps in one CUDA graph",
        "value": round(state_gbs, 1), "unit": "state GB/s", "us_per_step": round(ms * 1e3, 2),
        "gpu_launches": reps * steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm"], 4),
                     "traffic": ncu_traffic("kda_decode_kernel", DECODE_SOURCES),
                     "kernel": "kda_decode_kernel", "peak_source": pk["src"] + " burst copy",
                     "bytes_per_launch": n_units * DECODE_BYTES_PER_UNIT},
        "e2e": {"value": round(cx.ws * n_units * 2 * STATE_BYTES / (e2e_ms * 1e-3) / 1e9, 1),
                "unit": "state GB/s", "us_per_step": round(e2e_ms * 1e3, 2),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "H2D of step i+1 and D2H of step i-1 run beside step i (two buffer sets, "
                           "copy streams ordered by events); the state updates stay in order"},
        "clocks": clk.summary(),
        "multi_token": multi,
        "fused_prologue_epilogue": fused,
    }


def bench_prefill_workload(cx: Ctx, args, name: str, calls: int):
    """One of the larger prefill workloads (the packed varlen batch with start states, or the 1M-token
    sequence), device-resident, timed with CUDA events over `calls` calls after 2 warm-up calls."""
    torch = cx.torch
    import linear_attention_chunkwise_gb300 as kda
    from linear_attention_chunkwise_gb300 import synth

    c = synth.WORKLOADS[name]
    p = synth.prefill_inputs(synth.workload_lengths(name), c["H"], D, c["dtype"], c["lo"], c["s0_std"],
                             synth.workload_seed(name) + 1000 * cx.rank, cx.dev)
    T, N = p.total_tokens, len(p.lengths)
    o = torch.empty_like(p.q)
    sf = torch.empty((N, H, D, D), dtype=torch.float32, device=cx.dev)
    work = torch.empty(kda.kda_prefill_workspace_bytes(c["dtype"], N, T, H), dtype=torch.uint8, device=cx.dev)

    def call():
        kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, o=o, S_final=sf, workspace=work,
                        stream=cx.stream)

    for _ in range(2):
        call()
    cx.barrier()
    ev0, ev1 = cx.events()
    with ClockSampler(cx.dev) as clk:
        ev0.record(cx.stream)
        for _ in range(calls):
            call()
        ev1.record(cx.stream)
        cx.barrier()
    ms_local = ev0.elapsed_time(ev1) / calls
    ms = cx.max_over_ranks(ms_local)
    states = N * H * STATE_BYTES * (2 if p.S0 is not None else 1)  # S_final out (+ S0 in)
    bytes_per_call = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + states
    achieved = bytes_per_call / (ms_local * 1e-3) / 1e9
    flops = T * H * PREFILL_FLOPS_PER_TOKEN_HEAD
    pk = cx.peaks
    del work, o, sf, p
    torch.cuda.empty_cache()
    return {
        "workload": c["name"], "tokens": T, "sequences": N, "calls": calls,
        "value": round(whole_job_mtok_s(T, cx.ws, ms), 3), "unit": "Mtok/s", "ms_per_call": round(ms, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm"], 4), "traffic": None,
                     "kernel": "kda_prefill call (chunk table + chunk prep + scan kernels)",
                     "peak_source": pk["src"] + " burst copy", "bytes_per_launch": bytes_per_call},
        "tensor": {"achieved": round(flops / (ms_local * 1e-3) / 1e12, 2), "peak": pk["bf16"], "unit": "TFLOP/s",
                   "frac": round(flops / (ms_local * 1e-3) / 1e12 / pk["bf16"], 4)},
        "clocks": clk.summary(),
    }


def bench_prefill_fused(cx: Ctx, args):
    """The 8k prefill through kda_prefill_ex with every fusion: q/k L2 norm, sigmoid beta and the
    output RMSNorm x gate (one pass after the scan).  Device-resident inputs, CUDA events."""
    torch = cx.torch
    import linear_attention_chunkwise_gb300 as kda
    from linear_attention_chunkwise_gb300 import synth

    c = synth.WORKLOADS[PREFILL_WORKLOAD]
    p = synth.prefill_inputs(c["lengths"], c["H"], D, c["dtype"], c["lo"], c["s0_std"],
                             synth.workload_seed(PREFILL_WORKLOAD) + 1000 * cx.rank, cx.dev)
    T = p.total_tokens
    g = torch.Generator(device=cx.dev).manual_seed(7 + cx.rank)
    gate = torch.randn(p.q.shape, generator=g, device=cx.dev).to(p.q.dtype)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, out_gate=gate,
                    rms_weight=torch.ones(D, dtype=torch.float32, device=cx.dev))
    o = torch.empty_like(p.q)
    sf = torch.empty((1, H, D, D), dtype=torch.float32, device=cx.dev)
    work = torch.empty(kda.kda_prefill_workspace_bytes(torch.bfloat16, 1, T, H), dtype=torch.uint8, device=cx.dev)

    def call():
        kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, fusion=fz, o=o, S_final=sf,
                           workspace=work, stream=cx.stream)

    for _ in range(max(3, args.warmup)):
        call()
    cx.barrier()
    ev0, ev1 = cx.events()
    ev0.record(cx.stream)
    for _ in range(args.steps):
        call()
    ev1.record(cx.stream)
    cx.barrier()
    ms = cx.max_over_ranks(ev0.elapsed_time(ev1) / args.steps)
    return {"workload": "KDA chunkwise prefill B=1 H=32 T=8192 through kda_prefill_ex with L2-normalised q/k, "
                        "sigmoid beta and RMSNorm x output gate fused",
            "value": round(T * cx.ws / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s", "us_per_call": round(ms * 1e3, 1)}


def bench_backward(cx: Ctx, args):
    """Prefill backward on the 8k workload (grad_o ~ N(0,1) bf16, grad_S_final ~ N(0, 0.01)): one call
    reruns the chunkwise forward with a snapshot per chunk and walks every head back."""
    torch = cx.torch
    import linear_attention_chunkwise_gb300 as kda
    from linear_attention_chunkwise_gb300 import synth

    c = synth.WORKLOADS[PREFILL_WORKLOAD]
    p = synth.prefill_inputs(c["lengths"], c["H"], D, c["dtype"], c["lo"], c["s0_std"],
                             synth.workload_seed(PREFILL_WORKLOAD) + 1000 * cx.rank, cx.dev)
    T = p.total_tokens
    g = torch.Generator(device=cx.dev).manual_seed(11 + cx.rank)
    dO = torch.randn(p.q.shape, generator=g, device=cx.dev).to(p.q.dtype)
    dSf = torch.randn((1, H, D, D), generator=g, device=cx.dev) * 0.1
    f32 = dict(dtype=torch.float32, device=cx.dev)
    grads = (torch.empty((T, H, D), **f32), torch.empty((T, H, D), **f32), torch.empty((T, H, D), **f32),
             torch.empty((T, H, D), **f32), torch.empty((T, H), **f32), torch.empty((1, H, D, D), **f32))
    wsb = kda.kda_prefill_backward_workspace_bytes(torch.bfloat16, 1, T, H)
    work = torch.empty(wsb, dtype=torch.uint8, device=cx.dev)

    def call():
        kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, None, dSf, grads=grads,
                                 workspace=work, stream=cx.stream)

    n = max(3, min(args.steps, 10))
    for _ in range(max(3, args.warmup)):
        call()
    cx.barrier()
    ev0, ev1 = cx.events()
    with ClockSampler(cx.dev) as clk:
        ev0.record(cx.stream)
        for _ in range(n):
            call()
        ev1.record(cx.stream)
        cx.barrier()
    ms_local = ev0.elapsed_time(ev1) / n
    ms = cx.max_over_ranks(ms_local)
    bytes_per_call = T * H * BACKWARD_BYTES_PER_TOKEN_HEAD + 2 * H * STATE_BYTES  # + grad_S_final, grad_S0
    achieved = bytes_per_call / (ms_local * 1e-3) / 1e9
    flops_per_call = 2 * BACKWARD_MACS_PER_CHUNK_HEAD * (-(-T // 64)) * H
    achieved_tf = flops_per_call / (ms_local * 1e-3) / 1e12
    pk = cx.peaks
    del work

    # the same call through the fused prologue (q, k L2-normalised and beta = sigmoid(logits) inside,
    # the chain rule through both applied to the gradients): its two elementwise kernels on top
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=1e-6)
    work = torch.empty(kda.kda_prefill_backward_ex_workspace_bytes(torch.bfloat16, 1, T, H), dtype=torch.uint8,
                       device=cx.dev)

    def call_fused():
        kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, None, dSf, fusion=fz,
                                    grads=grads, workspace=work, stream=cx.stream)

    for _ in range(3):
        call_fused()
    ev0, ev1 = cx.events()
    ev0.record(cx.stream)
    for _ in range(n):
        call_fused()
    ev1.record(cx.stream)
    cx.stream.synchronize()
    ms_fused = ev0.elapsed_time(ev1) / n
    del work

    # through the output gate as well (kda_prefill_backward_gated): dL/dy in, dL/dgate and dL/dweight out
    gate = torch.randn(p.q.shape, generator=g, device=cx.dev).to(p.q.dtype)
    wrms = torch.ones(D, **f32)
    fzg = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=1e-6, out_gate=gate, rms_weight=wrms, rms_eps=1e-5)
    work = torch.empty(kda.kda_prefill_backward_gated_workspace_bytes(torch.bfloat16, 1, T, H), dtype=torch.uint8,
                       device=cx.dev)
    grads_g = grads + (torch.empty((T, H, D), **f32), torch.empty((D,), **f32))

    def call_gated():
        kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, None, dSf, fusion=fzg,
                                       grads=grads_g, workspace=work, stream=cx.stream)

    for _ in range(3):
        call_gated()
    ev0.record(cx.stream)
    for _ in range(n):
        call_gated()
    ev1.record(cx.stream)
    cx.stream.synchronize()
    ms_gated = ev0.elapsed_time(ev1) / n
    del work, grads, grads_g, gate
    # kernels per call: chunk table + snapshot entries, the internal forward (chunk table + its pass-1 and
    # scan launches; one sequence: no schedule kernel), then prep, adjoint scan and value+key
    sms = torch.cuda.get_device_properties(cx.dev).multi_processor_count
    n_prep, n_scan = piecewise_launches(-(-T // 64)) if 2 * H * 2 <= sms else (1, 1)
    launches = 2 + (1 + n_prep + n_scan) + 3
    return {
        "workload": "KDA prefill backward B=1 H=32 T=8192 d=128, bf16 q/k/v/grad_o, fp32 gates, S0=0, "
                    "grad_S_final given; fp32 gradients of q, k, v, log_alpha, beta, S0",
        "value": round(T * cx.ws / (ms * 1e-3) / 1e6, 3), "unit": "Mtok/s", "ms_per_call": round(ms, 3),
        "calls": n,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm"], 4),
                     "traffic": ncu_traffic("kda_prefill_backward", BACKWARD_SOURCES),
                     "kernel": "kda_prefill_backward call (chunkwise forward with per-chunk snapshots + "
                               "reverse walk)",
                     "peak_source": pk["src"] + " burst copy", "bytes_per_launch": bytes_per_call},
        "tensor": {"achieved": round(achieved_tf, 2), "peak": round(pk["bf16"] * TF32_OVER_BF16, 1),
                   "unit": "TFLOP/s", "frac": round(achieved_tf / (pk["bf16"] * TF32_OVER_BF16), 4),
                   "flops_per_launch": flops_per_call, "dtype": "tf32 (fp32 operands rounded), fp32 accumulate",
                   "peak_source": pk["src"] + " bf16 burst x nominal tf32/bf16 ratio 1.1/2.25"},
        "gpu_launches_per_call": launches,
        "fused_prologue": {"ms_per_call": round(ms_fused, 3), "gpu_launches_per_call": launches + 2,
                           "what": "kda_prefill_backward_ex, L2 norm of q, k and sigmoid beta fused"},
        "gated": {"ms_per_call": round(ms_gated, 3), "gpu_launches_per_call": launches + 4,
                  "what": "kda_prefill_backward_gated: the prologue and the output gate RMSNorm(o) x weight x gate "
                          "(dL/dgate, dL/dweight out)"},
        "clocks": clk.summary(),
    }


def run_ours(args):
    from linear_attention_chunkwise_gb300 import _build
    _build.build()
    cx = Ctx()
    pf = bench_prefill(cx, args) if args.only in ("all", "prefill") else None
    dc = bench_decode(cx, args) if args.only in ("all", "decode") else None
    bw = bench_backward(cx, args) if args.only in ("all", "backward") else None
    pfz = bench_prefill_fused(cx, args) if args.only == "prefill_fused" else None
    wl = {}
    if args.only in ("all", "prefill", "prefill_large"):
        wl["varlen_prefill"] = bench_prefill_workload(cx, args, "varlen_prefill", 5)
        wl["long_prefill_1m"] = bench_prefill_workload(cx, args, "long_prefill_1m", 3)
    out = {"metric": METRIC}
    if pf is not None:
        out.update({
            "value": round(pf["value"], 3), "unit": "Mtok/s", "n_gpus": cx.ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(pf["ms"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta sigmoid(N(0,1)), "
                    "log_alpha U[-0.2,0])",
            "config": {"workload": "KDA chunkwise prefill B=1 H=32 T=8192 dk=dv=128, bf16 q/k/v, "
                                   "fp32 gates and state, S0=0, chunk 64",
                       "tokens_per_step_per_gpu": pf["tokens"], "heads": H,
                       "l2": "inputs larger than L2 (404 MB read per step), no flush",
                       "parallelism": f"independent problem per GPU x{cx.ws}"},
            "roofline": pf["roofline"], "tensor": pf["tensor"], "e2e": pf["e2e"],
            "gpu_launches": pf["launches"], "clocks": pf["clocks"], "prefill_variants": pf["variants"],
            "chain_bound": pf["chain_bound"],
        })
    if dc is not None:
        out["decode"] = dc
    if bw is not None:
        out["backward"] = bw
    if pfz is not None:
        out["prefill_fused"] = pfz
    if wl:
        out["prefill_workloads"] = wl
    if cx.rank == 0 and not args.no_cpu_baseline and pf is not None:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if cx.rank == 0:
        print(json.dumps(out), flush=True)
    if cx.ws > 1:
        cx.dist.barrier()
        cx.dist.destroy_process_group()


# ------------------------------------------------------- oracle timing ----

def _oracle_inputs(tokens: int, seed: int):
    """The 8k prefill workload's inputs (or its first `tokens` tokens), generated on the CPU."""
    from linear_attention_chunkwise_gb300 import synth
    c = synth.WORKLOADS[PREFILL_WORKLOAD]
    pi = synth.prefill_inputs([tokens], c["H"], D, c["dtype"], c["lo"], None, seed, "cpu")
    f = lambda t: t.float().numpy()
    return f(pi.q), f(pi.k), f(pi.v), f(pi.log_alpha), f(pi.beta), [0, tokens]


def _time_oracle_runs(target_seconds: float, max_steps: int | None = None):
    """Time the oracle on the 8k workload: whole-workload passes repeated to fill
    about target_seconds, or a token prefix when one pass would take longer."""
    import oracle
    oracle.build()
    T = synth_tokens()
    q, k, v, la, b, _ = _oracle_inputs(T, seed=5)
    oracle.kda_prefill(q[:16], k[:16], v[:16], la[:16], b[:16], [0, 16], None)   # load, touch
    t0 = time.perf_counter()
    oracle.kda_prefill(q[:256], k[:256], v[:256], la[:256], b[:256], [0, 256], None)
    per_token = (time.perf_counter() - t0) / 256
    tokens = int(min(T, max(64, target_seconds / max(per_token, 1e-9))))
    reps = max(1, int(round(target_seconds / max(per_token * tokens, 1e-9))))
    if max_steps is not None:
        reps = max(1, min(reps, max_steps))
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.kda_prefill(q[:tokens], k[:tokens], v[:tokens], la[:tokens], b[:tokens], [0, tokens], None)
        times.append(time.perf_counter() - t0)
    return tokens, times, oracle.num_threads(0)


def synth_tokens() -> int:
    from linear_attention_chunkwise_gb300 import synth
    return int(synth.WORKLOADS[PREFILL_WORKLOAD]["lengths"][0])


def cpu_baseline(target_seconds: float):
    tokens, times, cores = _time_oracle_runs(target_seconds)
    total = sum(times)
    return {"value": round(len(times) * tokens / total / 1e6, 6), "unit": "Mtok/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{len(times)} pass(es) over {tokens} of the 8192 tokens x 32 heads of the 8k prefill "
                      f"workload, fp64 token loop, {total:.1f} s wall"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    # warm-up: one short untimed oracle call is made inside _time_oracle_runs
    tokens, times, cores = _time_oracle_runs(args.cpu_seconds / max(1, args.steps), max_steps=1)
    step_times = times
    for _ in range(args.steps - 1):
        step_times += _time_oracle_runs_fixed(tokens)
    s = sum(step_times) / len(step_times)
    value = tokens / s / 1e6
    out = {
        "metric": METRIC, "value": round(value, 6), "unit": "Mtok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(s * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": "KDA chunkwise prefill B=1 H=32 T=8192 dk=dv=128, bf16 q/k/v, fp32 gates and state, "
                               "S0=0, chunk 64", "sample_tokens_per_step": tokens, "heads": H},
        "cpu_baseline": {"value": round(value, 6), "unit": "Mtok/s", "cores": cores, "kind": "oracle",
                         "sample": f"{tokens} of the 8192 tokens x 32 heads per step, fp64 token loop"},
        "e2e": {"value": round(value, 6), "unit": "Mtok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def _time_oracle_runs_fixed(tokens: int):
    import oracle
    q, k, v, la, b, _ = _oracle_inputs(tokens, seed=5)
    t0 = time.perf_counter()
    oracle.kda_prefill(q, k, v, la, b, [0, tokens], None)
    return [time.perf_counter() - t0]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-reps", type=int, default=5, help="replays of the 100-step decode graph")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target wall time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "backward", "prefill_fused", "prefill_large"],
                    default="all",
                    help="profiling aid: run only one workload (the JSON line then lacks the other)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
