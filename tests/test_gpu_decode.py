"""GPU parity of kda_decode_step (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("permute", [False, True])
def test_decode_small_parity(dtype, permute):
    N, H, steps = 6, 3, 4
    slots = 9 if permute else N
    d = synth.decode_inputs(N, H, steps, dtype=dtype, seed=31, device="cuda", num_slots=slots,
                            permute_slots=permute)
    S_ref = host(d.S).astype(np.float64)
    S_before = d.S.clone()
    idx = None if d.state_indices is None else d.state_indices.cpu().numpy()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(steps):
        o = kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], d.S, d.state_indices,
                                device_status=status)
        o_ref = oracle.kda_decode_step(host(d.q[t]), host(d.k[t]), host(d.v[t]), host(d.log_alpha[t]),
                                       host(d.beta[t]), S_ref, idx)
        torch.cuda.synchronize()
        assert rell2(host(o), o_ref) < TOL
        # the state path is fp32 end to end: much tighter than the bf16 budget
        assert rell2(host(d.S), S_ref) < 1e-5
    assert int(status.item()) == 0
    if permute:
        named = set(idx.tolist())
        for s in range(slots):
            if s not in named:
                assert torch.equal(d.S[s], S_before[s]), "unnamed slot was touched"


def test_decode_bad_slot_is_reported_and_skipped():
    N, H = 4, 2
    d = synth.decode_inputs(N, H, 1, seed=5, device="cuda", num_slots=6, permute_slots=True)
    idx = torch.tensor([0, 7, 2, -1], dtype=torch.int32, device="cuda")
    S_before = d.S.clone()
    o = torch.full((N, H, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_decode_step(d.q[0], d.k[0], d.v[0], d.log_alpha[0], d.beta[0], d.S, idx, o=o, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_BAD_SLOT
    assert torch.all(o[1] == 3.0) and torch.all(o[3] == 3.0)     # skipped rows untouched
    for s in (1, 3, 4, 5):
        assert torch.equal(d.S[s], S_before[s])
    assert not torch.equal(d.S[0], S_before[0])


def test_decode_config3_graph_all_units():
    """256 sequences x 32 heads, 100 steps captured in one CUDA graph (the bench's launch
    configuration).  Every (sequence, head) unit is checked against the oracle, which runs the same
    100 steps on the exact input bytes: o of every step and the state after step 100.  The bound is
    applied to the whole tensors and to each unit on its own; the worst unit is printed."""
    c = synth.WORKLOADS["decode_256x32"]
    d = synth.workload_inputs("decode_256x32", device="cuda")
    N, H, steps = c["N"], c["H"], c["steps"]
    S_ref = host(d.S).astype(np.float64)  # [N, H, 128, 128], updated in place by the oracle
    o_all = torch.empty((steps, N, H, 128), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=stream):
        for t in range(steps):
            kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], d.S, None, o=o_all[t],
                                device_status=status)
    graph.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    err2 = np.zeros((N, H))  # per unit: squared error and squared reference norm of o over all steps
    ref2 = np.zeros((N, H))
    for t in range(steps):
        o_ref = oracle.kda_decode_step(host(d.q[t]), host(d.k[t]), host(d.v[t]), host(d.log_alpha[t]),
                                       host(d.beta[t]), S_ref)
        diff = host(o_all[t]).astype(np.float64) - o_ref
        err2 += np.sum(diff * diff, axis=-1)
        ref2 += np.sum(o_ref * o_ref, axis=-1)
    unit_o = np.sqrt(err2 / np.maximum(ref2, 1e-300))
    S_gpu = host(d.S).astype(np.float64)
    dS = S_gpu - S_ref
    unit_s = np.sqrt(np.sum(dS * dS, axis=(2, 3)) / np.maximum(np.sum(S_ref * S_ref, axis=(2, 3)), 1e-300))
    whole_o = float(np.sqrt(err2.sum() / ref2.sum()))
    whole_s = rell2(S_gpu, S_ref)
    wo = np.unravel_index(np.argmax(unit_o), unit_o.shape)
    ws = np.unravel_index(np.argmax(unit_s), unit_s.shape)
    print(f"decode 256x32x100: rel-L2 o {whole_o:.3e} (worst unit {tuple(int(x) for x in wo)}: "
          f"{unit_o[wo]:.3e}), S after step 100 {whole_s:.3e} (worst unit {tuple(int(x) for x in ws)}: "
          f"{unit_s[ws]:.3e})")
    assert whole_o < TOL and float(unit_o.max()) < TOL
    # the state path is fp32 end to end (bf16 only in the inputs): far inside the bf16 budget
    assert whole_s < 1e-4 and float(unit_s.max()) < 1e-4


# ------------------------------------------------------------ multi-token --

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_equals_single_steps(dtype):
    """T tokens in one launch == T single-step launches (same per-token arithmetic)."""
    N, H, T = 5, 3, 6
    d = synth.decode_inputs(N, H, T, dtype=dtype, seed=71, device="cuda", num_slots=8, permute_slots=True)
    S_single = d.S.clone()
    o_single = torch.stack([kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], S_single,
                                                d.state_indices) for t in range(T)], dim=1)
    tm = lambda x: x.transpose(0, 1).contiguous()  # [T, N, ...] -> [N, T, ...]
    S_multi = d.S.clone()
    o_multi, steps = kda.kda_decode_multi(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), S_multi,
                                          d.state_indices, return_steps=True)
    torch.cuda.synchronize()
    assert torch.equal(o_multi, o_single)
    assert torch.equal(S_multi, S_single)
    idx = d.state_indices.long()
    assert torch.equal(steps[:, -1], S_multi[idx])
    # state after token t == state after t+1 single steps
    S_ref = d.S.clone()
    for t in range(T):
        kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], S_ref, d.state_indices)
        torch.cuda.synchronize()
        assert torch.equal(steps[:, t], S_ref[idx])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_multi_many_units_equals_single_steps(dtype):
    """More (sequence, head) units than two per SM: each CTA walks several units with the next one's
    state and inputs prefetched; results stay bitwise equal to single steps, including a bad slot
    (flagged and skipped by both paths) and the per-token state output."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, T = 4, 4
    N = (2 * sms) // H + 37  # > 2 * SM count units, not a multiple of the grid
    d = synth.decode_inputs(N, H, T, dtype=dtype, seed=73, device="cuda", num_slots=N + 5, permute_slots=True)
    idx = d.state_indices.clone()
    idx[N // 3] = N + 5  # out of range
    st_s = torch.zeros(1, dtype=torch.int32, device="cuda")
    S_single = d.S.clone()
    o_single = torch.stack([kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], S_single, idx,
                                                device_status=st_s) for t in range(T)], dim=1)
    tm = lambda x: x.transpose(0, 1).contiguous()
    st_m = torch.zeros(1, dtype=torch.int32, device="cuda")
    S_multi = d.S.clone()
    o_multi, steps = kda.kda_decode_multi(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), S_multi, idx,
                                          device_status=st_m, return_steps=True)
    torch.cuda.synchronize()
    assert int(st_m.item()) == kda.KDA_DEV_BAD_SLOT and int(st_s.item()) == kda.KDA_DEV_BAD_SLOT
    ok = torch.ones(N, dtype=torch.bool, device="cuda")
    ok[N // 3] = False
    assert torch.equal(o_multi[ok], o_single[ok])
    assert torch.equal(S_multi, S_single)
    good = idx[ok].long()
    assert torch.equal(steps[ok][:, -1], S_multi[good])


def test_decode_multi_oracle_and_slots():
    N, H, T = 6, 4, 4
    d = synth.decode_inputs(N, H, T, seed=72, device="cuda", num_slots=10, permute_slots=True)
    S_before = d.S.clone()
    S_ref = host(d.S).astype(np.float64)
    idx = d.state_indices.cpu().numpy()
    o_ref = np.stack([oracle.kda_decode_step(host(d.q[t]), host(d.k[t]), host(d.v[t]), host(d.log_alpha[t]),
                                             host(d.beta[t]), S_ref, idx) for t in range(T)], axis=1)
    tm = lambda x: x.transpose(0, 1).contiguous()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o = kda.kda_decode_multi(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), d.S, d.state_indices,
                             device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert rell2(host(o), o_ref) < TOL
    assert rell2(host(d.S), S_ref) < 1e-5
    for s in set(range(10)) - set(idx.tolist()):
        assert torch.equal(d.S[s], S_before[s])


def test_decode_multi_equals_prefill():
    """T decode tokens == a prefill over the same T tokens from the same start state."""
    N, H, T = 3, 2, 70
    p = synth.prefill_inputs([T] * N, H, s0_std=0.02, seed=73, device="cuda")
    o_p, sf = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    S = p.S0.clone()
    r = lambda x: x.view(N, T, *x.shape[1:]).contiguous()
    o_m = kda.kda_decode_multi(r(p.q), r(p.k), r(p.v), r(p.log_alpha), r(p.beta), S)
    torch.cuda.synchronize()
    assert rell2(host(o_m.view_as(o_p)), host(o_p)) < TOL
    assert rell2(host(S), host(sf)) < TOL
