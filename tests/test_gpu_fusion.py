"""GPU parity of the fused prologue / epilogue (kda_prefill_ex, kda_decode_step_ex).

Inputs are raw (q, k not normalised, beta given as logits); the oracle applies
its plain definitions (oracle.l2_normalize, oracle.sigmoid,
oracle.rmsnorm_gate) to the exact input values, runs the recurrence in fp64,
and the GPU result must match within the rel-L2 bound.  The output gate in
prefill runs after the scan as one pass over o and the gate: covered on varlen
batches, a long single sequence (scan pieces) and the 8k workload.
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

L2_EPS, RMS_EPS = 1e-6, 1e-5


def _raw_inputs(lengths, H, dtype, seed):
    """Prefill inputs with un-normalised q, k (row scales 0.3 .. 3) and beta logits."""
    p = synth.prefill_inputs(lengths, H, dtype=dtype, s0_std=0.02, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 7)
    T = p.q.shape[0]
    sq = 0.3 + 2.7 * torch.rand((T, H, 1), generator=g, device="cuda")
    sk = 0.3 + 2.7 * torch.rand((T, H, 1), generator=g, device="cuda")
    p.q = (p.q.float() * sq).to(dtype)
    p.k = (p.k.float() * sk).to(dtype)
    p.beta = torch.randn((T, H), generator=g, device="cuda") * 1.5  # logits
    gate = torch.randn((T, H, 128), generator=g, device="cuda").to(dtype)
    w = 1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")
    return p, gate, w


def _oracle(p, gate, w, heads, prologue=True, epilogue=True):
    cu = p.cu_seqlens.cpu().tolist()
    hidx = torch.tensor(heads, dtype=torch.long, device="cuda")
    outs, finals = [], []
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        sl = lambda t: host(t[a:b].index_select(1, hidx))
        q, k, beta = sl(p.q), sl(p.k), sl(p.beta)
        if prologue:
            q, k, beta = oracle.l2_normalize(q, L2_EPS), oracle.l2_normalize(k, L2_EPS), oracle.sigmoid(beta)
        S0 = None if p.S0 is None else host(p.S0[n].index_select(0, hidx))[None]
        o, sf = oracle.kda_prefill(q, k, sl(p.v), sl(p.log_alpha), beta, [0, b - a], S0)
        if epilogue:
            o = oracle.rmsnorm_gate(o, sl(gate), host(w), RMS_EPS)
        outs.append(o)
        finals.append(sf[0])
    return outs, finals


def _check(p, o, sf, outs, finals, heads):
    cu = p.cu_seqlens.cpu().tolist()
    hidx = torch.tensor(heads, dtype=torch.long, device="cuda")
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if b > a:
            assert rell2(host(o[a:b].index_select(1, hidx)), outs[n]) < TOL, n
        assert rell2(host(sf[n].index_select(0, hidx)), finals[n]) < TOL, n


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("epilogue", [False, True])
def test_prefill_fused_varlen(dtype, epilogue):
    p, gate, w = _raw_inputs([130, 0, 7, 64, 300, 1, 129], 3, dtype, 621)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate if epilogue else None,
                    rms_weight=w, rms_eps=RMS_EPS)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, sf = kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, fusion=fz,
                               device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    outs, finals = _oracle(p, gate, w, [0, 1, 2], epilogue=epilogue)
    _check(p, o, sf, outs, finals, [0, 1, 2])


def test_prefill_output_gate_alone_matches_plain_prefill():
    # epilogue only: the state path is untouched, so S_final equals kda_prefill's bit for bit
    p = synth.prefill_inputs([500, 77], 2, s0_std=0.02, seed=622, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    gate = torch.randn(p.q.shape, generator=g, device="cuda").to(p.q.dtype)
    o_ref, sf_ref = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    o, sf = kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0,
                               fusion=kda.Fusion(out_gate=gate, rms_eps=RMS_EPS))
    torch.cuda.synchronize()
    assert torch.equal(sf, sf_ref)
    # y from the fused path vs RMSNorm x gate applied to kda_prefill's bf16 o: two bf16 roundings apart,
    # each with relative RMS error about 2^-8 / sqrt(3) = 2.3e-3, so about 3.2e-3 together
    y_ref = oracle.rmsnorm_gate(host(o_ref), host(gate), None, RMS_EPS)
    assert rell2(host(o), y_ref) < 5e-3


def test_prefill_fused_long_sequence_pieces():
    L = 64 * 64 + 200  # the scan runs in two pieces; the output gate pairs the two dv slices
    p, gate, w = _raw_inputs([L], 2, torch.bfloat16, 623)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w,
                    rms_eps=RMS_EPS)
    o, sf = kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, fusion=fz)
    torch.cuda.synchronize()
    outs, finals = _oracle(p, gate, w, [0, 1])
    _check(p, o, sf, outs, finals, [0, 1])


def test_prefill_fused_8k_workload():
    p = synth.workload_inputs("prefill_8k", device="cuda")
    g = torch.Generator(device="cuda").manual_seed(624)
    T, H, _ = p.q.shape
    p.q = (p.q.float() * 1.7).to(p.q.dtype)
    p.beta = torch.randn((T, H), generator=g, device="cuda")
    gate = torch.randn((T, H, 128), generator=g, device="cuda").to(p.q.dtype)
    w = 1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w,
                    rms_eps=RMS_EPS)
    o, sf = kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, fusion=fz)
    torch.cuda.synchronize()
    heads = [5, 30]
    outs, finals = _oracle(p, gate, w, heads)
    _check(p, o, sf, outs, finals, heads)


def test_prefill_fusion_needs_the_two_pass_workspace():
    p, gate, w = _raw_inputs([100], 1, torch.bfloat16, 625)
    small = torch.empty(max(kda.kda_prefill_min_workspace_bytes(kda.KDA_DTYPE_BF16, 1, 100, 1), 256),
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, fusion=kda.Fusion(l2norm_qk=True),
                           workspace=small)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("flags", [(True, True, True), (True, False, False), (False, True, False),
                                   (False, False, True)])
def test_decode_fused_steps(dtype, flags):
    l2n, sig, og = flags
    N, H, steps = 6, 3, 4
    d = synth.decode_inputs(N, H, steps, dtype=dtype, seed=626, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(627)
    d.q = (d.q.float() * (0.3 + 2.7 * torch.rand(d.q.shape[:-1] + (1,), generator=g, device="cuda"))).to(dtype)
    d.k = (d.k.float() * (0.3 + 2.7 * torch.rand(d.k.shape[:-1] + (1,), generator=g, device="cuda"))).to(dtype)
    beta = torch.randn(d.beta.shape, generator=g, device="cuda") if sig else d.beta
    gate = torch.randn(d.q.shape, generator=g, device="cuda").to(dtype)
    w = 1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")
    S_ref = host(d.S).astype(np.float64)
    idx = None if d.state_indices is None else d.state_indices.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(steps):
        fz = kda.Fusion(l2norm_qk=l2n, beta_sigmoid=sig, l2_eps=L2_EPS, out_gate=gate[t] if og else None,
                        rms_weight=w, rms_eps=RMS_EPS)
        o = kda.kda_decode_step_ex(d.q[t], d.k[t], d.v[t], d.log_alpha[t], beta[t], d.S, d.state_indices,
                                   fusion=fz, device_status=status)
        q, k, b = host(d.q[t]), host(d.k[t]), host(beta[t])
        if l2n:
            q, k = oracle.l2_normalize(q, L2_EPS), oracle.l2_normalize(k, L2_EPS)
        if sig:
            b = oracle.sigmoid(b)
        o_ref = oracle.kda_decode_step(q, k, host(d.v[t]), host(d.log_alpha[t]), b, S_ref, idx)
        if og:
            o_ref = oracle.rmsnorm_gate(o_ref, host(gate[t]), host(w), RMS_EPS)
        torch.cuda.synchronize()
        assert rell2(host(o), o_ref) < TOL, t
        assert rell2(host(d.S), S_ref) < 1e-4, t
    assert int(status.item()) == 0


def test_decode_multi_fused_many_units():
    """The fused multi-token path with more units than two per SM (prefetched units, T = 3)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, T = 2, 3
    N = sms + 17
    d = synth.decode_inputs(N, H, T, seed=631, device="cuda", num_slots=N + 2, permute_slots=True)
    g = torch.Generator(device="cuda").manual_seed(632)
    scale = lambda x: (x.float() * (0.3 + 2.7 * torch.rand(x.shape[:-1] + (1,), generator=g, device="cuda"))).to(
        torch.bfloat16)
    q, k = scale(d.q), scale(d.k)
    beta = torch.randn(d.beta.shape, generator=g, device="cuda")
    gate = torch.randn(d.q.shape, generator=g, device="cuda").to(torch.bfloat16)
    tm = lambda x: x.transpose(0, 1).contiguous()
    S_ref = host(d.S).astype(np.float64)
    idx = d.state_indices.cpu().numpy()
    o_ref = []
    for t in range(T):
        qq, kk = oracle.l2_normalize(host(q[t]), L2_EPS), oracle.l2_normalize(host(k[t]), L2_EPS)
        ot = oracle.kda_decode_step(qq, kk, host(d.v[t]), host(d.log_alpha[t]), oracle.sigmoid(host(beta[t])), S_ref,
                                    idx)
        o_ref.append(oracle.rmsnorm_gate(ot, host(gate[t]), np.ones(128), RMS_EPS))
    o_ref = np.stack(o_ref, axis=1)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=tm(gate), rms_eps=RMS_EPS)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.kda_decode_multi_ex(tm(q), tm(k), tm(d.v), tm(d.log_alpha), tm(beta), d.S, d.state_indices, fusion=fz,
                                device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rell2(host(o), o_ref) < TOL
    assert rell2(host(d.S), S_ref) < 1e-4


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_fused(dtype):
    N, H, T = 5, 3, 11  # two token batches in the kernel (8 + 3)
    d = synth.decode_inputs(N, H, T, dtype=dtype, seed=628, device="cuda", num_slots=7, permute_slots=True)
    g = torch.Generator(device="cuda").manual_seed(629)
    scale = lambda x: (x.float() * (0.3 + 2.7 * torch.rand(x.shape[:-1] + (1,), generator=g, device="cuda"))).to(dtype)
    q, k = scale(d.q), scale(d.k)
    beta = torch.randn(d.beta.shape, generator=g, device="cuda")
    gate = torch.randn(d.q.shape, generator=g, device="cuda").to(dtype)
    w = 1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")
    tm = lambda x: x.transpose(0, 1).contiguous()  # [T, N, ...] -> [N, T, ...]
    S_ref = host(d.S).astype(np.float64)
    idx = d.state_indices.cpu().numpy()
    o_ref = []
    for t in range(T):
        qq, kk = oracle.l2_normalize(host(q[t]), L2_EPS), oracle.l2_normalize(host(k[t]), L2_EPS)
        ot = oracle.kda_decode_step(qq, kk, host(d.v[t]), host(d.log_alpha[t]), oracle.sigmoid(host(beta[t])), S_ref,
                                    idx)
        o_ref.append(oracle.rmsnorm_gate(ot, host(gate[t]), host(w), RMS_EPS))
    o_ref = np.stack(o_ref, axis=1)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=tm(gate), rms_weight=w,
                    rms_eps=RMS_EPS)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.kda_decode_multi_ex(tm(q), tm(k), tm(d.v), tm(d.log_alpha), tm(beta), d.S, d.state_indices, fusion=fz,
                                device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rell2(host(o), o_ref) < TOL
    assert rell2(host(d.S), S_ref) < 1e-4


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_fused_prologue_only(dtype):
    """Prologue fusions without the output gate, with the per-step states."""
    N, H, T = 6, 3, 10  # two token batches in the kernel (8 + 2)
    d = synth.decode_inputs(N, H, T, dtype=dtype, seed=630, device="cuda", num_slots=9, permute_slots=True)
    g = torch.Generator(device="cuda").manual_seed(631)
    scale = lambda x: (x.float() * (0.3 + 2.7 * torch.rand(x.shape[:-1] + (1,), generator=g, device="cuda"))).to(dtype)
    q, k = scale(d.q), scale(d.k)
    beta = torch.randn(d.beta.shape, generator=g, device="cuda")
    tm = lambda x: x.transpose(0, 1).contiguous()  # [T, N, ...] -> [N, T, ...]
    S_ref = host(d.S).astype(np.float64)
    idx = d.state_indices.cpu().numpy()
    o_ref = []
    for t in range(T):
        qq, kk = oracle.l2_normalize(host(q[t]), L2_EPS), oracle.l2_normalize(host(k[t]), L2_EPS)
        o_ref.append(oracle.kda_decode_step(qq, kk, host(d.v[t]), host(d.log_alpha[t]),
                                            oracle.sigmoid(host(beta[t])), S_ref, idx))
    o_ref = np.stack(o_ref, axis=1)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS)
    S_steps = torch.empty((N, T, H, 128, 128), dtype=torch.float32, device="cuda")
    o, steps = kda.kda_decode_multi_ex(tm(q), tm(k), tm(d.v), tm(d.log_alpha), tm(beta), d.S, d.state_indices,
                                       fusion=fz, S_steps=S_steps, return_steps=True)
    torch.cuda.synchronize()
    assert rell2(host(o), o_ref) < TOL
    assert rell2(host(d.S), S_ref) < 1e-4
    # the last step's state is the state written back
    assert torch.equal(steps[:, T - 1], d.S[d.state_indices.long()])


def test_prefill_fused_one_set_scan_grid():
    # more scan CTAs (sequences x heads x 2) than SMs: the scan's one-operand-set form, two CTAs per SM,
    # with the fused prologue in pass 1 and the output gate after the scan
    lengths = [130, 0, 7, 64, 300, 1, 129, 65, 513, 63, 200, 33]
    H = torch.cuda.get_device_properties(0).multi_processor_count // (2 * len(lengths)) + 1
    p, gate, w = _raw_inputs(lengths, H, torch.bfloat16, 631)
    fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, l2_eps=L2_EPS, out_gate=gate, rms_weight=w, rms_eps=RMS_EPS)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, sf = kda.kda_prefill_ex(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, fusion=fz,
                               device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    heads = [0, H // 2, H - 1]
    outs, finals = _oracle(p, gate, w, heads)
    _check(p, o, sf, outs, finals, heads)
