"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method itself: it only draws the
random inputs (and L2-normalises q and k, which the library takes as a
caller precondition).  Both the CUDA path and the fp64 oracle are fed from
here; neither computes its inputs from the other.

Recipe (the synthetic workloads of the prefill / decode benchmarks):
  * q, k ~ N(0, 1) in fp32, L2-normalised over the 128 channels of each
    (token, head), then cast to the input dtype;
  * v ~ N(0, 1), cast to the input dtype;
  * beta = sigmoid(N(0, 1)) in fp32, one per (token, head);
  * log_alpha ~ U[lo, 0] in fp32, one per (token, head, channel);
  * S0 ~ N(0, std^2) in fp32 per (sequence, head) when a start state is used.
Draw order: q, k, v, beta, log_alpha, S0; one torch.Generator on the target
device seeded with ``seed``.  Large tensors are drawn in token slabs so the
fp32 temporaries stay bounded; the slab size is part of the recipe.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SLAB_TOKENS = 65536

# The five workloads, by name: tiny fp32 prefill, 8k prefill, packed varlen
# prefill with start states, 256 x 32-head decode, and the 1M-token prefill.
WORKLOADS = {
    "tiny_prefill": dict(kind="prefill", name="tiny prefill B=1 H=2 T=256 d=128 fp32", seed=20260, lengths=[256],
                         H=2, dtype=torch.float32, lo=-0.2, s0_std=None),
    "prefill_8k": dict(kind="prefill", name="prefill B=1 H=32 T=8192 d=128 bf16", seed=20261, lengths=[8192], H=32,
                       dtype=torch.bfloat16, lo=-0.2, s0_std=None),
    "varlen_prefill": dict(kind="prefill", name="varlen prefill N=16 len~U[1024,65536] H=32 d=128 bf16, S0~N(0,0.02)",
                           seed=20262, lengths=None, num_seqs=16, len_lo=1024, len_hi=65536, H=32,
                           dtype=torch.bfloat16, lo=-0.2, s0_std=0.02),
    "decode_256x32": dict(kind="decode", name="decode N=256 H=32 d=128 bf16, 100 steps, S~N(0,0.02)", seed=20263,
                          N=256, H=32, steps=100, dtype=torch.bfloat16, lo=-0.2, s_std=0.02),
    "long_prefill_1m": dict(kind="prefill", name="long prefill B=1 H=32 T=1048576 d=128 bf16", seed=20264,
                            lengths=[1048576], H=32, dtype=torch.bfloat16, lo=-0.05, s0_std=None),
}


def workload_seed(name: str) -> int:
    return int(WORKLOADS[name]["seed"])


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> list[int]:
    """Sequence lengths ~ U{lo..hi} (inclusive), drawn on the CPU so every device agrees."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (num_seqs,), generator=g)]


def workload_lengths(name: str) -> list[int]:
    c = WORKLOADS[name]
    if c.get("lengths") is not None:
        return list(c["lengths"])
    return varlen_lengths(c["num_seqs"], c["len_lo"], c["len_hi"], workload_seed(name) + 7)


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, d] dtype
    k: torch.Tensor            # [T, H, d] dtype
    v: torch.Tensor            # [T, H, d] dtype
    beta: torch.Tensor         # [T, H] fp32
    log_alpha: torch.Tensor    # [T, H, d] fp32
    S0: torch.Tensor | None    # [N, H, d, d] fp32
    cu_seqlens: torch.Tensor   # [N+1] int32, same device
    lengths: list[int]

    @property
    def total_tokens(self) -> int:
        return int(self.q.shape[0])


def _unit_rows(shape, g, dtype, device, slab):
    """N(0,1) rows L2-normalised over the last dim, drawn slab by slab over dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    for s in range(0, shape[0], slab):
        e = min(shape[0], s + slab)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
        out[s:e] = x.to(dtype)
    return out


def _normal(shape, g, dtype, device, slab, std=1.0):
    out = torch.empty(shape, dtype=dtype, device=device)
    for s in range(0, shape[0], slab):
        e = min(shape[0], s + slab)
        x = torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        out[s:e] = (x * std).to(dtype)
    return out


def _sigmoid_normal(shape, g, device, slab):
    out = torch.empty(shape, dtype=torch.float32, device=device)
    for s in range(0, shape[0], slab):
        e = min(shape[0], s + slab)
        out[s:e] = torch.sigmoid(torch.randn((e - s,) + tuple(shape[1:]), generator=g, device=device))
    return out


def _uniform(shape, g, device, slab, lo, hi):
    out = torch.empty(shape, dtype=torch.float32, device=device)
    for s in range(0, shape[0], slab):
        e = min(shape[0], s + slab)
        out[s:e] = torch.rand((e - s,) + tuple(shape[1:]), generator=g, device=device) * (hi - lo) + lo
    return out


def prefill_inputs(lengths, H: int, d: int = 128, dtype=torch.bfloat16, lo: float = -0.2,
                   s0_std: float | None = None, seed: int = 0, device="cuda",
                   slab: int = SLAB_TOKENS) -> PrefillInputs:
    lengths = [int(x) for x in lengths]
    T = sum(lengths)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = _unit_rows((T, H, d), g, dtype, device, slab)
    k = _unit_rows((T, H, d), g, dtype, device, slab)
    v = _normal((T, H, d), g, dtype, device, slab)
    beta = _sigmoid_normal((T, H), g, device, slab)
    log_alpha = _uniform((T, H, d), g, device, slab, lo, 0.0)
    S0 = None
    if s0_std is not None:
        S0 = _normal((len(lengths), H, d, d), g, torch.float32, device, slab, std=s0_std)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    cu_seqlens = torch.tensor(cu, dtype=torch.int32, device=device)
    return PrefillInputs(q, k, v, beta, log_alpha, S0, cu_seqlens, lengths)


@dataclass
class DecodeInputs:
    q: torch.Tensor          # [steps, N, H, d]
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor       # [steps, N, H] fp32
    log_alpha: torch.Tensor  # [steps, N, H, d] fp32
    S: torch.Tensor          # [slots, H, d, d] fp32
    state_indices: torch.Tensor | None  # [N] int32 or None


def decode_inputs(N: int, H: int, steps: int, d: int = 128, dtype=torch.bfloat16, lo: float = -0.2,
                  s_std: float = 0.02, seed: int = 0, device="cuda", num_slots: int | None = None,
                  permute_slots: bool = False) -> DecodeInputs:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    shp = (steps * N, H, d)
    q = _unit_rows(shp, g, dtype, device, SLAB_TOKENS).view(steps, N, H, d)
    k = _unit_rows(shp, g, dtype, device, SLAB_TOKENS).view(steps, N, H, d)
    v = _normal(shp, g, dtype, device, SLAB_TOKENS).view(steps, N, H, d)
    beta = _sigmoid_normal((steps * N, H), g, device, SLAB_TOKENS).view(steps, N, H)
    log_alpha = _uniform(shp, g, device, SLAB_TOKENS, lo, 0.0).view(steps, N, H, d)
    slots = N if num_slots is None else int(num_slots)
    S = _normal((slots, H, d, d), g, torch.float32, device, 64, std=s_std)
    idx = None
    if permute_slots or slots != N:
        gc = torch.Generator(device="cpu")
        gc.manual_seed(int(seed) + 1)
        idx = torch.randperm(slots, generator=gc)[:N].to(torch.int32).to(device)
    return DecodeInputs(q, k, v, beta, log_alpha, S, idx)


def workload_inputs(name: str, device="cuda"):
    c = WORKLOADS[name]
    if c["kind"] == "prefill":
        return prefill_inputs(workload_lengths(name), c["H"], 128, c["dtype"], c["lo"], c["s0_std"],
                              workload_seed(name), device)
    return decode_inputs(c["N"], c["H"], c["steps"], 128, c["dtype"], c["lo"], c["s_std"],
                         workload_seed(name), device)
