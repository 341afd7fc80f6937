"""GPU parity of kda_prefill (through the C ABI) against the fp64 oracle.

Small cases span several chunks and ragged tails; the five benchmark
workloads run at full size in the launch configuration the bench times (the
two-pass path), the oracle checking all heads (8k prefill), sampled heads per
sequence (varlen) or two sampled heads over the full length (1M tokens).
Both prefill paths (two-pass and single-pass, chosen by workspace size) are
checked on the small and edge cases.
"""
import numpy as np
import pytest
import torch

import oracle
import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, oracle_prefill_heads, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


PATHS = ["two_pass", "single_pass"]


def run_gpu(p, **kw):
    status = torch.zeros(1, dtype=torch.int32, device=p.q.device)
    o, sf = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, device_status=status, **kw)
    torch.cuda.synchronize()
    return o, sf, int(status.item())


def check_against_oracle(p, o, sf, heads_per_seq=None, tol=TOL):
    cu = p.cu_seqlens.cpu().tolist()
    errs = []
    for n, (heads, o_ref, s_ref) in enumerate(oracle_prefill_heads(p, heads_per_seq)):
        a, b = cu[n], cu[n + 1]
        hidx = torch.tensor(heads, dtype=torch.long, device=o.device)
        if b > a:
            eo = rell2(host(o[a:b].index_select(1, hidx)), o_ref)
            assert eo < tol, f"seq {n}: o rel-L2 {eo}"
            errs.append(eo)
        es = rell2(host(sf[n].index_select(0, hidx)), s_ref)
        assert es < tol, f"seq {n}: S_final rel-L2 {es}"
    return errs


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("lengths", [[1], [63], [64], [65], [200], [1000]])
def test_prefill_single_sequence(lengths, path):
    p = synth.prefill_inputs(lengths, 3, seed=sum(lengths), device="cuda")
    o, sf, st = run_gpu(p, path=path)
    assert st == 0
    check_against_oracle(p, o, sf)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_prefill_varlen_with_states(dtype, path):
    lengths = [130, 0, 7, 64, 300, 1, 129]
    p = synth.prefill_inputs(lengths, 4, dtype=dtype, s0_std=0.02, seed=17, device="cuda")
    o, sf, st = run_gpu(p, path=path)
    assert st == 0
    check_against_oracle(p, o, sf)
    # the empty sequence returns its start state bit for bit
    assert torch.equal(sf[1], p.S0[1])


@pytest.mark.parametrize("path", PATHS)
def test_prefill_identity_gates_keep_state_exactly(path):
    """beta = 0, alpha = 1: every chunk is the identity on S (fp32 path, exact)."""
    p = synth.prefill_inputs([70, 200], 2, s0_std=0.5, seed=3, device="cuda")
    p.beta.zero_()
    p.log_alpha.zero_()
    o, sf, st = run_gpu(p, path=path)
    assert st == 0
    assert torch.equal(sf, p.S0)


def test_prefill_split_invariant():
    """prefill(A || B) == prefill(B, S0 = S_final(A)) (prefix-cache boundary)."""
    p = synth.prefill_inputs([777], 2, s0_std=0.02, seed=8, device="cuda")
    o, sf, _ = run_gpu(p)
    c = 300
    sl = lambda t, a, b: t[a:b].contiguous()
    cu_a = torch.tensor([0, c], dtype=torch.int32, device="cuda")
    cu_b = torch.tensor([0, 777 - c], dtype=torch.int32, device="cuda")
    oa, sa = kda.kda_prefill(sl(p.q, 0, c), sl(p.k, 0, c), sl(p.v, 0, c), sl(p.log_alpha, 0, c),
                             sl(p.beta, 0, c), cu_a, p.S0)
    ob, sb = kda.kda_prefill(sl(p.q, c, 777), sl(p.k, c, 777), sl(p.v, c, 777), sl(p.log_alpha, c, 777),
                             sl(p.beta, c, 777), cu_b, sa)
    torch.cuda.synchronize()
    assert rell2(host(torch.cat([oa, ob])), host(o)) < TOL
    assert rell2(host(sb), host(sf)) < TOL


def test_prefill_equals_decode_steps():
    """The two execution modes agree: prefill over n tokens == n decode steps."""
    n_tok, H = 70, 2
    p = synth.prefill_inputs([n_tok], H, s0_std=0.02, seed=21, device="cuda")
    o, sf, _ = run_gpu(p)
    S = p.S0.clone()
    outs = []
    for t in range(n_tok):
        sl = lambda x: x[t:t + 1].contiguous()
        outs.append(kda.kda_decode_step(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha), sl(p.beta), S))
    torch.cuda.synchronize()
    assert rell2(host(torch.cat(outs)), host(o)) < TOL
    assert rell2(host(S), host(sf)) < TOL


@pytest.mark.parametrize("path", PATHS)
def test_prefill_deterministic_and_in_bounds(path):
    p = synth.prefill_inputs([333, 64, 5], 3, s0_std=0.02, seed=4, device="cuda")
    T, H = p.q.shape[:2]
    pad = 4096
    o_buf = torch.full((T * H * 128 + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = o_buf[pad:pad + T * H * 128].view(T, H, 128)
    sf_buf = torch.full((3 * H * 128 * 128 + 2 * pad,), 9.0, dtype=torch.float32, device="cuda")
    sf = sf_buf[pad:pad + 3 * H * 128 * 128].view(3, H, 128, 128)
    kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, o=o, S_final=sf, path=path)
    o1, sf1 = o.clone(), sf.clone()
    kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, o=o, S_final=sf, path=path)
    torch.cuda.synchronize()
    assert torch.equal(o, o1) and torch.equal(sf, sf1)
    assert torch.all(o_buf[:pad] == 7.0) and torch.all(o_buf[-pad:] == 7.0)
    assert torch.all(sf_buf[:pad] == 9.0) and torch.all(sf_buf[-pad:] == 9.0)


@pytest.mark.parametrize("path", PATHS)
def test_prefill_bad_cu_seqlens_reported(path):
    p = synth.prefill_inputs([100, 50], 2, seed=2, device="cuda")
    p.cu_seqlens.copy_(torch.tensor([0, 120, 110], dtype=torch.int32))   # decreasing, wrong total
    o = torch.full_like(p.q, 5.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, None, o=o, device_status=status, path=path)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_BAD_CU_SEQLENS
    assert torch.all(o[120:] == 5.0)        # the malformed sequence wrote nothing


def test_prefill_config0_tiny_fp32():
    p = synth.workload_inputs("tiny_prefill", device="cuda")
    o, sf, st = run_gpu(p)
    assert st == 0 and o.dtype == torch.float32
    check_against_oracle(p, o, sf)


@pytest.mark.parametrize("path", PATHS)
def test_prefill_config1_all_heads(path):
    p = synth.workload_inputs("prefill_8k", device="cuda")
    o, sf, st = run_gpu(p, path=path)
    assert st == 0
    errs = check_against_oracle(p, o, sf)
    assert max(errs) < TOL


def test_prefill_config2_varlen_sampled_heads():
    p = synth.workload_inputs("varlen_prefill", device="cuda")
    o, sf, st = run_gpu(p)
    assert st == 0
    N, H = len(p.lengths), p.q.shape[1]
    g = torch.Generator().manual_seed(2026)
    heads = [sorted(torch.randperm(H, generator=g)[:4].tolist()) for _ in range(N)]
    check_against_oracle(p, o, sf, heads)


@pytest.mark.slow
def test_prefill_config4_long_two_heads():
    p = synth.workload_inputs("long_prefill_1m", device="cuda")
    o, sf, st = run_gpu(p)
    assert st == 0
    g = torch.Generator().manual_seed(4)
    heads = [sorted(torch.randperm(p.q.shape[1], generator=g)[:2].tolist())]
    check_against_oracle(p, o, sf, heads)


@pytest.mark.parametrize("alias", [False, True])
def test_prefill_piecewise_two_sequences(alias):
    # two sequences of different lengths, few heads: the scan runs piecewise (pass 1 ahead of it
    # on another stream); the short sequence ends inside the first piece, the long one spans four.
    # With alias, S_final is S0 itself (the carry between pieces then lives in S0's memory).
    p = synth.prefill_inputs([7000, 3500], 4, s0_std=0.02, seed=631, device="cuda")
    S0_copy = p.S0.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sf_out = p.S0 if alias else None
    o, sf = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, S_final=sf_out,
                            device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    p.S0 = S0_copy  # the oracle starts from the original states
    check_against_oracle(p, o, sf, [[0, 3], [1, 2]])
    # without S_final the pieces carry the state in the workspace instead: the same o
    o1, _ = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, S0_copy, return_final=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o1)


def test_prefill_in_cuda_graph():
    # under stream capture the library runs one prep + one scan on the capturing stream (no
    # library-owned stream); the replayed graph gives the eager result bit for bit
    p = synth.prefill_inputs([5000, 300], 2, s0_std=0.02, seed=641, device="cuda")
    o_ref, sf_ref = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    T, H, _ = p.q.shape
    ws = torch.empty(kda.kda_prefill_workspace_bytes(torch.bfloat16, 2, T, H), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(o_ref)
    sf = torch.empty_like(sf_ref)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, o=o, S_final=sf, workspace=ws,
                        stream=s)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(sf, sf_ref)
