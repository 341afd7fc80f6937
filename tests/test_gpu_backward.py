"""GPU parity of kda_prefill_backward against the fp64 oracle gradient.

The oracle's gradient (oracle.kda_prefill_backward) is itself pinned by
finite differences of the forward oracle (tests/test_oracle_backward_pins.py).
Here the CUDA path is compared with it element by element, all six gradients
(q, k, v, log_alpha, beta, S0) at rel-L2 <= 1e-2, on the same seeded inputs:
varlen batches with empty, one-token and ragged sequences; several head
counts; fp32 and bf16 inputs; no grad_S_final; bitwise repeatability; and the
8k-token 32-head workload on two sampled heads (heads are independent, so the oracle on
those heads alone gives their exact gradients).  The same for the backward through
the fused prologue (kda_prefill_backward_ex) and through the output gate
(kda_prefill_backward_gated: eight gradients, the gate's and the RMSNorm weight's
included, against oracle.kda_prefill_backward_gated, itself pinned by finite
differences in tests/test_oracle_gate_pins.py).
"""
import numpy as np
import pytest
import torch

import oracle
import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

NAMES = ("q", "k", "v", "log_alpha", "beta", "S0")


def _cotangents(p, seed, with_final=True):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    T, H, d = p.q.shape
    dO = torch.randn((T, H, d), generator=g, device="cuda").to(p.q.dtype)
    dSf = None
    if with_final:
        dSf = torch.randn((len(p.lengths), H, d, d), generator=g, device="cuda") * 0.1
    return dO, dSf


def _oracle(p, dO, dSf, heads=None):
    """Oracle gradients (float64) over all or some heads of every sequence."""
    hidx = torch.arange(p.q.shape[1], device="cuda") if heads is None else torch.tensor(heads, device="cuda")
    sel = lambda t: None if t is None else host(t.index_select(1, hidx))
    return oracle.kda_prefill_backward(sel(p.q), sel(p.k), sel(p.v), sel(p.log_alpha), sel(p.beta),
                                       p.cu_seqlens.cpu().numpy(), sel(p.S0), sel(dO), sel(dSf))


def _gpu(p, dO, dSf, status=None):
    out = kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf,
                                   device_status=status)
    torch.cuda.synchronize()
    return out


def _compare(got, ref, heads=None, tol=TOL):
    for name, g, r in zip(NAMES, got, ref):
        g = host(g if heads is None else g.index_select(1, torch.tensor(heads, device=g.device)))
        assert np.all(np.isfinite(g)), name
        if np.linalg.norm(r) == 0:
            assert np.abs(g).max() == 0, name
            continue
        err = rell2(g, r)
        assert err <= tol, (name, err)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_backward_varlen_matches_oracle(dtype):
    lengths = [300, 0, 64, 1, 129, 200]
    p = synth.prefill_inputs(lengths, H=2, dtype=dtype, s0_std=0.02, seed=41)
    dO, dSf = _cotangents(p, 42)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu(p, dO, dSf, status)
    assert int(status.item()) == 0
    _compare(got, _oracle(p, dO, dSf))


@pytest.mark.parametrize("H", [1, 5, 40])
def test_backward_head_counts(H):
    p = synth.prefill_inputs([150], H=H, s0_std=0.02, seed=43 + H)
    dO, dSf = _cotangents(p, 44)
    _compare(_gpu(p, dO, dSf), _oracle(p, dO, dSf))


def test_backward_without_final_gradient_or_S0():
    p = synth.prefill_inputs([70, 190], H=3, seed=45)
    dO, _ = _cotangents(p, 46, with_final=False)
    got = kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, None, None,
                                   need_grad_S0=False)
    torch.cuda.synchronize()
    assert got[5] is None
    ref = _oracle(p, dO, None)
    _compare(got[:5], ref[:5])


def test_backward_no_tokens_passes_final_gradient_through():
    p = synth.prefill_inputs([0, 0], H=2, s0_std=0.02, seed=47)
    dO = torch.empty((0, 2, 128), dtype=p.q.dtype, device="cuda")
    dSf = torch.randn((2, 2, 128, 128), device="cuda")
    got = _gpu(p, dO, dSf)
    assert torch.equal(got[5], dSf)
    assert all(g.numel() == 0 for g in got[:5])


def test_backward_is_deterministic():
    """No atomics anywhere: two calls give identical bits."""
    p = synth.prefill_inputs([100, 300], H=4, s0_std=0.02, seed=48)
    dO, dSf = _cotangents(p, 49)
    a = _gpu(p, dO, dSf)
    b = _gpu(p, dO, dSf)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_8k_sampled_heads():
    """The 8192-token, 32-head bf16 workload, as the bench runs it; heads 0 and 31 against the oracle."""
    p = synth.prefill_inputs([8192], H=32, seed=synth.workload_seed("prefill_8k"))
    dO, dSf = _cotangents(p, 50)
    got = _gpu(p, dO, dSf)
    heads = [0, 31]
    _compare(got, _oracle(p, dO, dSf, heads), heads)


def test_backward_degenerate_gates():
    """Tokens with beta = 0 (no write: du still drives dbeta) and log_alpha = 0 (no decay)."""
    p = synth.prefill_inputs([200, 90], H=2, s0_std=0.02, seed=51)
    p.beta[::7] = 0.0
    p.log_alpha[::5] = 0.0
    dO, dSf = _cotangents(p, 52)
    _compare(_gpu(p, dO, dSf), _oracle(p, dO, dSf))


def test_backward_strong_decay():
    """log_alpha ~ U[-1, 0]: per-chunk gate spans up to e^{32} around the reference row."""
    p = synth.prefill_inputs([256, 77], H=2, lo=-1.0, s0_std=0.02, seed=53)
    dO, dSf = _cotangents(p, 54)
    _compare(_gpu(p, dO, dSf), _oracle(p, dO, dSf))


def test_backward_in_cuda_graph():
    """The whole backward call (its chunkwise forward included) captures into a CUDA graph and
    replays bit for bit like the eager call."""
    p = synth.prefill_inputs([700, 130], H=2, s0_std=0.02, seed=55)
    dO, dSf = _cotangents(p, 56)
    ref = _gpu(p, dO, dSf)
    T, H, _ = p.q.shape
    ws = torch.empty(kda.kda_prefill_backward_workspace_bytes(p.q.dtype, 2, T, H), dtype=torch.uint8, device="cuda")
    grads = tuple(torch.empty_like(x) for x in ref)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf, grads=grads,
                                 workspace=ws, stream=s)
    for x in grads:
        x.zero_()
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip(grads, ref):
        assert torch.equal(x, y)


# ------------------------------------------------------------- fused prologue --
L2_EPS = 1e-6


def _raw(lengths, H, dtype, seed):
    """Inputs as kda_prefill_ex takes them raw: q, k rows scaled by U[0.3, 3], beta as N(0, 1.5^2) logits."""
    p = synth.prefill_inputs(lengths, H=H, dtype=dtype, s0_std=0.02, seed=seed)
    g = torch.Generator(device="cuda")
    g.manual_seed(seed + 7)
    T = p.q.shape[0]
    p.q = (p.q.float() * (0.3 + 2.7 * torch.rand((T, H, 1), generator=g, device="cuda"))).to(dtype)
    p.k = (p.k.float() * (0.3 + 2.7 * torch.rand((T, H, 1), generator=g, device="cuda"))).to(dtype)
    p.beta = torch.randn((T, H), generator=g, device="cuda") * 1.5
    return p


def _fused_oracle(p, dO, dSf, l2norm_qk, beta_sigmoid):
    return oracle.kda_prefill_backward_fused(host(p.q), host(p.k), host(p.v), host(p.log_alpha), host(p.beta),
                                             p.cu_seqlens.cpu().numpy(), host(p.S0), host(dO),
                                             None if dSf is None else host(dSf), l2norm_qk=l2norm_qk,
                                             beta_sigmoid=beta_sigmoid, l2_eps=L2_EPS)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_backward_fused_prologue_matches_oracle(dtype):
    p = _raw([300, 0, 64, 1, 129, 200], H=2, dtype=dtype, seed=61)
    dO, dSf = _cotangents(p, 62)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS)
    got = kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf, fusion=fz,
                                      device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare(got, _fused_oracle(p, dO, dSf, True, True))


@pytest.mark.parametrize("l2norm_qk,beta_sigmoid", [(True, False), (False, True)])
def test_backward_fused_prologue_single_flags(l2norm_qk, beta_sigmoid):
    p = _raw([190, 70], H=3, dtype=torch.bfloat16, seed=63)
    if not l2norm_qk:  # the plain recurrence wants unit-norm q, k
        p.q = torch.nn.functional.normalize(p.q.float(), dim=-1).to(p.q.dtype)
        p.k = torch.nn.functional.normalize(p.k.float(), dim=-1).to(p.k.dtype)
    if not beta_sigmoid:
        p.beta = torch.sigmoid(p.beta)
    dO, dSf = _cotangents(p, 64)
    fz = kda.Fusion(l2norm_qk=l2norm_qk, beta_sigmoid=beta_sigmoid, l2_eps=L2_EPS)
    got = kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf, fusion=fz)
    torch.cuda.synchronize()
    _compare(got, _fused_oracle(p, dO, dSf, l2norm_qk, beta_sigmoid))


def test_backward_ex_without_flags_is_the_plain_backward():
    p = synth.prefill_inputs([100, 250], H=2, s0_std=0.02, seed=65)
    dO, dSf = _cotangents(p, 66)
    a = _gpu(p, dO, dSf)
    b = kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf,
                                    fusion=kda.Fusion())
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_backward_ex_rejects_the_output_gate():
    p = _raw([64], H=1, dtype=torch.bfloat16, seed=67)
    dO, _ = _cotangents(p, 68, with_final=False)
    fz = kda.Fusion(l2norm_qk=True, out_gate=torch.ones_like(p.q))
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_backward_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, fusion=fz)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED


# ---------------------------------------------------------------- output gate --
RMS_EPS = 1e-5
GATED_NAMES = NAMES + ("out_gate", "rms_weight")


def _gate(p, seed, weight=True):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    T, H, d = p.q.shape
    gate = torch.randn((T, H, d), generator=g, device="cuda").to(p.q.dtype)
    w = (1.0 + 0.5 * torch.randn(d, generator=g, device="cuda")) if weight else None
    return gate, w


def _gated_oracle(p, dY, dSf, gate, w, l2norm_qk, beta_sigmoid, heads=None):
    """Oracle gradients of the gated output; w None is passed as ones so that dL/dweight comes back."""
    hidx = torch.arange(p.q.shape[1], device="cuda") if heads is None else torch.tensor(heads, device="cuda")
    sel = lambda t: None if t is None else host(t.index_select(1, hidx))
    return oracle.kda_prefill_backward_gated(sel(p.q), sel(p.k), sel(p.v), sel(p.log_alpha), sel(p.beta),
                                             p.cu_seqlens.cpu().numpy(), sel(p.S0), sel(dY), sel(dSf), sel(gate),
                                             np.ones(128) if w is None else host(w), RMS_EPS, l2norm_qk=l2norm_qk,
                                             beta_sigmoid=beta_sigmoid, l2_eps=L2_EPS)


def _compare_gated(got, ref, heads=None, tol=TOL, with_dw=True):
    _compare(got[:6], ref[:6], heads, tol)
    g = host(got[6] if heads is None else got[6].index_select(1, torch.tensor(heads, device=got[6].device)))
    assert np.all(np.isfinite(g))
    assert rell2(g, ref[6]) <= tol, ("out_gate", rell2(g, ref[6]))
    if with_dw:
        assert rell2(host(got[7]), ref[7]) <= tol, ("rms_weight", rell2(host(got[7]), ref[7]))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_backward_gated_matches_oracle(dtype):
    """Prologue and output gate together, varlen with empty, one-token and ragged sequences."""
    p = _raw([300, 0, 64, 1, 129, 200], H=2, dtype=dtype, seed=71)
    dY, dSf = _cotangents(p, 72)
    gate, w = _gate(p, 73)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w, rms_eps=RMS_EPS)
    got = kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dY, p.S0, dSf,
                                         fusion=fz, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _compare_gated(got, _gated_oracle(p, dY, dSf, gate, w, True, True))


def test_backward_gated_plain_inputs_unit_weight():
    """Output gate alone (q, k unit-norm, beta in (0, 1)), rms_weight NULL = ones, no grad_S_final."""
    p = synth.prefill_inputs([190, 70, 5], H=3, s0_std=0.02, seed=74)
    dY, _ = _cotangents(p, 75, with_final=False)
    gate, _ = _gate(p, 76, weight=False)
    fz = kda.Fusion(out_gate=gate, rms_eps=RMS_EPS)
    got = kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dY, p.S0, None,
                                         fusion=fz)
    torch.cuda.synchronize()
    _compare_gated(got, _gated_oracle(p, dY, None, gate, None, False, False))


def test_backward_gated_is_deterministic_and_skips_weight():
    p = _raw([500, 77], H=4, dtype=torch.bfloat16, seed=77)
    dY, dSf = _cotangents(p, 78)
    gate, w = _gate(p, 79)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w, rms_eps=RMS_EPS)
    run = lambda need_w: kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dY,
                                                        p.S0, dSf, fusion=fz, need_grad_rms_weight=need_w)
    a, b, c = run(True), run(True), run(False)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert c[7] is None
    for x, y in zip(a[:7], c[:7]):
        assert torch.equal(x, y)


def test_backward_gated_no_tokens():
    """No tokens: the gate's gradients are empty, dL/dweight is zero, grad_S0 is grad_S_final carried back."""
    p = synth.prefill_inputs([0, 0], H=2, s0_std=0.02, seed=80)
    dY = torch.empty((0, 2, 128), dtype=p.q.dtype, device="cuda")
    dSf = torch.randn((2, 2, 128, 128), device="cuda")
    gate = torch.empty((0, 2, 128), dtype=p.q.dtype, device="cuda")  # NULL pointer: allowed without tokens
    w = torch.ones(128, device="cuda")
    fz = kda.Fusion(out_gate=gate, rms_weight=w, rms_eps=RMS_EPS)
    got = kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dY, p.S0, dSf,
                                         fusion=fz)
    torch.cuda.synchronize()
    assert got[6].numel() == 0
    assert torch.equal(got[7], torch.zeros(128, device="cuda"))
    assert torch.equal(got[5], dSf)


def test_backward_gated_8k_sampled_heads():
    """The 8192-token, 32-head bf16 workload with prologue and gate; heads 0 and 31 against the oracle
    (dL/dweight sums over every head, so it is checked on the 4-head case above, not here)."""
    p = _raw([8192], H=32, dtype=torch.bfloat16, seed=81)
    dY, dSf = _cotangents(p, 82)
    gate, w = _gate(p, 83)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w, rms_eps=RMS_EPS)
    got = kda.kda_prefill_backward_gated(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dY, p.S0, dSf,
                                         fusion=fz)
    torch.cuda.synchronize()
    heads = [0, 31]
    _compare_gated(got, _gated_oracle(p, dY, dSf, gate, w, True, True, heads), heads, with_dw=False)


def test_backward_one_set_forward_grid():
    # more scan CTAs than SMs: the internal forward (a snapshot after every chunk) runs the scan's
    # one-operand-set form, two CTAs per SM; three sampled heads against the oracle
    lengths = [130, 0, 7, 64, 300, 1, 129, 65, 513, 63, 200, 33]
    H = torch.cuda.get_device_properties(0).multi_processor_count // (2 * len(lengths)) + 1
    p = synth.prefill_inputs(lengths, H=H, s0_std=0.02, seed=91)
    dO, dSf = _cotangents(p, 92)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _gpu(p, dO, dSf, status)
    assert int(status.item()) == 0
    heads = [0, H // 2, H - 1]
    _compare(got, _oracle(p, dO, dSf, heads), heads)
