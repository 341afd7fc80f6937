"""GPU parity of the scan's two buffering forms.

A scan grid that fits the GPU at one CTA per SM (few sequences x heads) runs with two operand sets
per CTA; a larger grid runs with one set, two CTAs per SM.  Both forms do the same arithmetic in the
same order, so a sequence's outputs do not depend on the form: a batch large enough for the one-set
form is checked against the fp64 oracle on every head, and each of its sequences, run alone (a grid
small enough for the two-set form), must give the same bits.
"""
import pytest
import torch

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, oracle_prefill_heads, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

# ragged lengths: one token, a chunk minus / plus one, an empty sequence, several chunks
LENGTHS = [1, 63, 64, 65, 130, 200, 0, 7, 300, 129, 513, 1000]


def _heads_for_one_set(n_seqs):
    """Heads per sequence so that the scan grid (sequences x heads x 2 slices) exceeds the SM count."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms // (2 * n_seqs) + 1


def _alone(p, n, fn):
    """fn(q, k, v, log_alpha, beta, cu_seqlens, S0) on sequence n by itself."""
    a, b = int(p.cu_seqlens[n].item()), int(p.cu_seqlens[n + 1].item())
    cu = torch.tensor([0, b - a], dtype=torch.int32, device="cuda")
    sl = lambda t: t[a:b].contiguous()
    S0 = None if p.S0 is None else p.S0[n:n + 1].contiguous()
    return fn(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha), sl(p.beta), cu, S0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_one_set_scan_matches_oracle_and_two_set_form(dtype):
    H = _heads_for_one_set(len(LENGTHS))
    p = synth.prefill_inputs(LENGTHS, H, dtype=dtype, s0_std=0.02, seed=1201, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, sf = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    cu = p.cu_seqlens.cpu().tolist()
    for n, (heads, o_ref, s_ref) in enumerate(oracle_prefill_heads(p)):
        a, b = cu[n], cu[n + 1]
        if b > a:
            assert rell2(host(o[a:b]), o_ref) < TOL, f"seq {n}: o"
        assert rell2(host(sf[n]), s_ref) < TOL, f"seq {n}: S_final"
    for n in range(len(LENGTHS)):  # the same sequence in a two-set grid: the same bits
        o1, sf1 = _alone(p, n, lambda *x: kda.kda_prefill(*x))
        torch.cuda.synchronize()
        a, b = cu[n], cu[n + 1]
        assert torch.equal(o1, o[a:b]), f"seq {n}: o differs between the scan forms"
        assert torch.equal(sf1[0], sf[n]), f"seq {n}: S_final differs between the scan forms"


def test_one_set_scan_snapshots():
    H = _heads_for_one_set(len(LENGTHS))
    p = synth.prefill_inputs(LENGTHS, H, s0_std=0.02, seed=1202, device="cuda")
    # a state after every chunk boundary inside each sequence and at each sequence end
    entries = []
    for n, L in enumerate(LENGTHS):
        entries += [(n, q) for q in list(range(64, L, 64)) + ([L] if L > 0 else [])]
    seq = torch.tensor([s for s, _ in entries], dtype=torch.int32, device="cuda")
    pos = torch.tensor([q for _, q in entries], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, sf, ss = kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, p.S0,
                                          device_status=status)
    o_ref, sf_ref = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(o, o_ref) and torch.equal(sf, sf_ref)
    cu = p.cu_seqlens.cpu().tolist()
    for i, (n, q) in enumerate(entries):
        # the prefix of sequence n alone (a two-set grid): its final state is the snapshot, bit for bit
        a = cu[n]
        cu1 = torch.tensor([0, q], dtype=torch.int32, device="cuda")
        sl = lambda t: t[a:a + q].contiguous()
        _, sfq = kda.kda_prefill(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha), sl(p.beta), cu1,
                                 p.S0[n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert torch.equal(ss[i], sfq[0]), f"snapshot {i} (sequence {n}, position {q})"
