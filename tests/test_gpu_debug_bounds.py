"""Bounds-checked build: every derived range stays inside its buffer on the test workloads.

A second copy of the library is built with KDA_DEBUG_BOUNDS.  In it, every CTA of the prefill (pass 1,
scan, single-pass), the backward (prep, adjoint scan, value, key, snapshot entries) checks, before it
touches memory, the ranges it derives from cu_seqlens, the schedule, the chunk table and the snapshot
entries: sequence and head in range, its chunks inside the workspace's images / records / snapshots,
its tokens inside [0, total_tokens), its snapshot entries inside the entry list.  A range outside its
buffer would set KDA_DEV_BOUNDS and skip that work (no trap).  The decode kernels derive no index from
the inputs but the slot, which every build checks (KDA_DEV_BAD_SLOT).

Each case runs the same call through the release library and the checked one: the status words must
match and carry no KDA_DEV_BOUNDS, and every output must be bitwise equal (the checks change nothing
when nothing is out of range).  The cases cover the layouts the kernels index differently: packed
varlen batches with empty and one-token sequences, scan grids of one and two CTAs per SM, the
piecewise schedule of long sequences, the
single-pass path, snapshots, the fused prologue and the output gate, decode with permuted
and bad slots, multi-token decode over several token batches, the backward (plain, fused, gated),
and a malformed cu_seqlens.
"""
import contextlib
import os

import pytest
import torch

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import _binding, _build, synth
from tests.conftest import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

DBG_DIR = os.path.join(_build.BUILD_DIR, "debug_bounds")


@pytest.fixture(scope="module")
def libs():
    path = _build.build(extra_flags=["-DKDA_DEBUG_BOUNDS"], lib_path=os.path.join(DBG_DIR, "libkda_debug_bounds.so"),
                        build_dir=DBG_DIR)
    return _binding.load_library(), _binding.load_library(path)


@contextlib.contextmanager
def _using(lib):
    saved = _binding._lib
    _binding._lib = lib
    try:
        yield
    finally:
        _binding._lib = saved


def _both(libs, fn):
    """fn(status) -> tuple of output tensors, run through the release and the checked library."""
    outs = []
    for lib in libs:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        with _using(lib):
            res = fn(status)
        torch.cuda.synchronize()
        outs.append((int(status.item()), [t for t in res if t is not None]))
    (s_rel, r_rel), (s_dbg, r_dbg) = outs
    assert s_dbg == s_rel, (s_rel, s_dbg)
    assert not (s_dbg & kda.KDA_DEV_BOUNDS)
    assert len(r_rel) == len(r_dbg)
    for a, b in zip(r_rel, r_dbg):
        assert torch.equal(a, b)
    return s_rel


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_prefill_varlen(libs, dtype, path):
    p = synth.prefill_inputs([300, 0, 64, 1, 129, 200], 2, dtype=dtype, s0_std=0.02, seed=901, device="cuda")
    st = _both(libs, lambda s: kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                                               device_status=s, path=path))
    assert st == 0


def test_prefill_one_set_scan(libs):
    # more scan CTAs than SMs: the one-operand-set scan, two CTAs per SM, plain and with snapshots
    lengths = [300, 0, 64, 1, 129, 200, 65, 63, 513, 7, 1000, 130]
    H = torch.cuda.get_device_properties(0).multi_processor_count // (2 * len(lengths)) + 1
    p = synth.prefill_inputs(lengths, H, s0_std=0.02, seed=907, device="cuda")
    assert _both(libs, lambda s: kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                                                 device_status=s)) == 0
    seq = torch.tensor([0, 0, 3, 4, 8, 8, 10, 11], dtype=torch.int32, device="cuda")
    pos = torch.tensor([64, 300, 1, 129, 448, 513, 1000, 64], dtype=torch.int32, device="cuda")
    assert _both(libs, lambda s: kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq,
                                                           pos, p.S0, device_status=s)) == 0


def test_prefill_piecewise_long_sequences(libs):
    p = synth.prefill_inputs([6000, 3100], 2, s0_std=0.02, seed=902, device="cuda")
    assert _both(libs, lambda s: kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                                                 device_status=s)) == 0


def test_prefill_snapshots(libs):
    p = synth.prefill_inputs([700, 64, 5, 1000], 2, s0_std=0.02, seed=903, device="cuda")
    seq = torch.tensor([0, 0, 0, 1, 2, 3, 3], dtype=torch.int32, device="cuda")
    pos = torch.tensor([64, 640, 700, 64, 5, 512, 1000], dtype=torch.int32, device="cuda")
    assert _both(libs, lambda s: kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq,
                                                           pos, p.S0, device_status=s)) == 0


def test_prefill_fused_prologue_and_output_gate(libs):
    p = synth.prefill_inputs([300, 77, 0, 4100], 2, s0_std=0.02, seed=904, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(905)
    gate = torch.randn(p.q.shape, generator=g, device="cuda").to(p.q.dtype)
    w = 1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=1e-6, out_gate=gate, rms_weight=w, rms_eps=1e-5)
    assert _both(libs, lambda s: kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                                                    fusion=fz, device_status=s)) == 0


def test_prefill_malformed_cu_seqlens(libs):
    p = synth.prefill_inputs([100, 100], 2, seed=906, device="cuda")
    bad = torch.tensor([0, 150, 120], dtype=torch.int32, device="cuda")  # decreasing, ends below T = 200
    st = _both(libs, lambda s: kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, bad, None,
                                               o=torch.zeros_like(p.q), return_final=False, device_status=s))
    assert st == kda.KDA_DEV_BAD_CU_SEQLENS


def test_decode_slots(libs):
    N, H, T = 37, 4, 11  # multi-token: two token batches per unit in the kernel
    d = synth.decode_inputs(N, H, T, seed=907, device="cuda", num_slots=N + 3, permute_slots=True)
    idx = d.state_indices.clone()
    idx[5] = N + 3  # out of range: flagged and skipped by every build
    tm = lambda x: x.transpose(0, 1).contiguous()

    # outputs start zeroed: the bad slot's rows are left as they are
    def step(s):
        S = d.S.clone()
        o = kda.kda_decode_step(d.q[0], d.k[0], d.v[0], d.log_alpha[0], d.beta[0], S, idx,
                                o=torch.zeros_like(d.v[0]), device_status=s)
        return o, S

    def multi(s):
        S = d.S.clone()
        steps = torch.zeros((N, T, H, 128, 128), device="cuda")
        o = kda.kda_decode_multi(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), S, idx,
                                 o=torch.zeros_like(tm(d.v)), S_steps=steps, device_status=s)
        return o, S, steps

    assert _both(libs, step) == kda.KDA_DEV_BAD_SLOT
    assert _both(libs, multi) == kda.KDA_DEV_BAD_SLOT


def test_backward_plain_fused_gated(libs):
    p = synth.prefill_inputs([300, 0, 64, 1, 129], 2, s0_std=0.02, seed=908, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(909)
    dO = torch.randn(p.q.shape, generator=g, device="cuda").to(p.q.dtype)
    dSf = torch.randn((5, 2, 128, 128), generator=g, device="cuda") * 0.1
    gate = torch.randn(p.q.shape, generator=g, device="cuda").to(p.q.dtype)
    assert _both(libs, lambda s: kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO,
                                                          p.S0, dSf, device_status=s)) == 0
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=1e-6)
    assert _both(libs, lambda s: kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO,
                                                             p.S0, dSf, fusion=fz, device_status=s)) == 0
    fz = kda.Fusion(out_gate=gate, rms_eps=1e-5)
    assert _both(libs, lambda s: kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens,
                                                                dO, p.S0, dSf, fusion=fz, device_status=s)) == 0
