"""GPU parity of kda_prefill_snapshots: states recorded at prefix boundaries.

The state after the first `pos` tokens of a sequence is, by definition, the
final state of a prefill over that prefix alone (the prefix-cache reading of
"Kimi Delta Attention (KDA)" (codewithdark), "KV Caching Challenges & vLLM
Contribution").  Each recorded state is checked against the fp64 oracle run
on the prefix, and against the GPU's own S_final of a prefill over the prefix
(same chunks, same arithmetic: bit-identical).  o and S_final of the call must
equal those of kda_prefill.  Invalid entries raise KDA_DEV_BAD_SNAPSHOT and
never disturb the valid ones.
"""
import pytest
import torch

import oracle
import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def _snap_tensors(entries):
    seq = torch.tensor([s for s, _ in entries], dtype=torch.int32, device="cuda")
    pos = torch.tensor([q for _, q in entries], dtype=torch.int32, device="cuda")
    return seq, pos


def _oracle_prefix_state(p, n, pos, heads):
    a = int(p.cu_seqlens[n].item())
    hidx = torch.tensor(heads, dtype=torch.long, device=p.q.device)
    sl = lambda t: host(t[a:a + pos].index_select(1, hidx))
    S0 = None if p.S0 is None else host(p.S0[n].index_select(0, hidx))[None]
    _, sf = oracle.kda_prefill(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha),
                               host(p.beta[a:a + pos].index_select(1, hidx)), [0, pos], S0)
    return sf[0]


def _gpu_prefix_state(p, n, pos):
    a = int(p.cu_seqlens[n].item())
    cu = torch.tensor([0, pos], dtype=torch.int32, device="cuda")
    S0 = None if p.S0 is None else p.S0[n:n + 1].contiguous()
    sl = lambda t: t[a:a + pos].contiguous()
    _, sf = kda.kda_prefill(sl(p.q), sl(p.k), sl(p.v), sl(p.log_alpha), sl(p.beta), cu, S0)
    return sf[0]


def _run(p, entries):
    seq, pos = _snap_tensors(entries)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, sf, ss = kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, p.S0,
                                          device_status=status)
    torch.cuda.synchronize()
    return o, sf, ss, int(status.item())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_snapshots_varlen_match_oracle_prefixes(dtype):
    lengths = [300, 0, 64, 1000, 129]
    p = synth.prefill_inputs(lengths, 3, dtype=dtype, s0_std=0.02, seed=611, device="cuda")
    entries = [(0, 64), (0, 256), (0, 300), (2, 64), (3, 128), (3, 640), (3, 1000), (4, 64), (4, 128), (4, 129)]
    o, sf, ss, st = _run(p, entries)
    assert st == 0
    o_ref, sf_ref = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    assert torch.equal(o, o_ref) and torch.equal(sf, sf_ref)
    for i, (n, pos) in enumerate(entries):
        ref = _oracle_prefix_state(p, n, pos, [0, 1, 2])
        assert rell2(host(ss[i]), ref) < TOL, (n, pos)
        assert torch.equal(ss[i], _gpu_prefix_state(p, n, pos)), (n, pos)
    # an entry at the sequence end is that sequence's S_final
    assert torch.equal(ss[2], sf[0]) and torch.equal(ss[6], sf[3]) and torch.equal(ss[9], sf[4])


def test_snapshots_across_pieces_of_a_long_sequence():
    # one sequence, two heads: 129 chunks, so the scan runs in three pieces of 43 chunks
    # (2752 tokens); entries sit on both sides of both piece boundaries and at the ragged end
    L = 64 * 64 * 2 + 37
    p = synth.prefill_inputs([L], 2, s0_std=0.02, seed=612, device="cuda")
    entries = [(0, 64), (0, 2688), (0, 2752), (0, 2816), (0, 4096), (0, 5440), (0, 5504), (0, 5568), (0, 8192),
               (0, L)]
    o, sf, ss, st = _run(p, entries)
    assert st == 0
    for i, (n, pos) in enumerate(entries):
        ref = _oracle_prefix_state(p, n, pos, [0, 1])
        assert rell2(host(ss[i]), ref) < TOL, pos
        assert torch.equal(ss[i], _gpu_prefix_state(p, n, pos)), pos
    assert torch.equal(ss[-1], sf[0])


def test_snapshots_on_the_8k_workload():
    # full-size 8k prefill (B=1, H=32, T=8192) with a state every 1024 tokens, in the
    # launch configuration the bench times; the oracle checks two sampled heads
    p = synth.workload_inputs("prefill_8k", device="cuda")
    entries = [(0, 1024 * i) for i in range(1, 9)]
    o, sf, ss, st = _run(p, entries)
    assert st == 0
    heads = [3, 29]
    hidx = torch.tensor(heads, dtype=torch.long, device="cuda")
    for i, (n, pos) in enumerate(entries[:2] + entries[-1:]):
        j = entries.index((n, pos))
        ref = _oracle_prefix_state(p, n, pos, heads)
        assert rell2(host(ss[j].index_select(0, hidx)), ref) < TOL, pos
    assert torch.equal(ss[-1], sf[0])
    assert torch.equal(ss[3], _gpu_prefix_state(p, 0, 4096))


def test_bad_snapshot_entries_are_flagged_and_skipped():
    lengths = [300, 200]
    p = synth.prefill_inputs(lengths, 2, seed=613, device="cuda")
    # (0, 100) is not chunk-aligned; (1, 256) is past the end; the rest are valid
    entries = [(0, 64), (0, 100), (0, 128), (1, 64), (1, 256)]
    seq, pos = _snap_tensors(entries)
    ss = torch.full((len(entries), 2, 128, 128), 7.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, S_snap=ss,
                              device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kda.KDA_DEV_BAD_SNAPSHOT
    for i in (0, 2, 3):
        n, q = entries[i]
        assert torch.equal(ss[i], _gpu_prefix_state(p, n, q))
    assert bool((ss[1] == 7.0).all()) and bool((ss[4] == 7.0).all())
    # unsorted and out-of-range sequence entries set the flag too
    for bad in ([(1, 64), (0, 64)], [(2, 64)], [(0, 0)]):
        seq, pos = _snap_tensors(bad)
        status.zero_()
        kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & kda.KDA_DEV_BAD_SNAPSHOT, bad


def test_snapshots_need_the_two_pass_workspace():
    p = synth.prefill_inputs([100], 1, seed=614, device="cuda")
    seq, pos = _snap_tensors([(0, 64)])
    small = torch.empty(max(kda.kda_prefill_min_workspace_bytes(kda.KDA_DTYPE_BF16, 1, 100, 1), 256),
                        dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, workspace=small)
