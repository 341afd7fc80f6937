"""Out-of-bounds write checks: every output buffer sits inside a larger allocation whose head and
tail are filled with a sentinel, the call writes through a view of the middle, and the sentinels
must survive.  Covers the decode state and o (single and multi-token, with the per-token states),
the prefill's state snapshots and the six gradients of the prefill backward; the prefill's own o
and S_final are covered in test_gpu_prefill.py."""
import pytest
import torch

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

PAD = 4096  # elements of sentinel on each side (keeps the 16-byte alignment of the view)


def _padded(shape, dtype, sentinel):
    n = 1
    for x in shape:
        n *= x
    buf = torch.full((n + 2 * PAD,), sentinel, dtype=dtype, device="cuda")
    return buf, buf[PAD:PAD + n].view(*shape)


def _intact(buf, sentinel):
    return bool(torch.all(buf[:PAD] == sentinel)) and bool(torch.all(buf[-PAD:] == sentinel))


def test_decode_step_writes_inside_its_buffers():
    N, H, slots = 5, 3, 9
    d = synth.decode_inputs(N, H, 2, seed=901, device="cuda", num_slots=slots, permute_slots=True)
    S_buf, S = _padded(d.S.shape, torch.float32, 9.0)
    S.copy_(d.S)
    o_buf, o = _padded((N, H, 128), torch.bfloat16, 7.0)
    for t in range(2):
        kda.kda_decode_step(d.q[t], d.k[t], d.v[t], d.log_alpha[t], d.beta[t], S, d.state_indices, o=o)
    torch.cuda.synchronize()
    assert _intact(S_buf, 9.0) and _intact(o_buf, 7.0)


@pytest.mark.parametrize("fused", [False, True])
def test_decode_multi_writes_inside_its_buffers(fused):
    N, H, T, slots = 4, 3, 5, 7
    d = synth.decode_inputs(N, H, T, seed=902, device="cuda", num_slots=slots, permute_slots=True)
    tm = lambda x: x.transpose(0, 1).contiguous()
    S_buf, S = _padded(d.S.shape, torch.float32, 9.0)
    S.copy_(d.S)
    o_buf, o = _padded((N, T, H, 128), torch.bfloat16, 7.0)
    st_buf, st = _padded((N, T, H, 128, 128), torch.float32, 5.0)
    if fused:
        gate = torch.randn((N, T, H, 128), device="cuda").to(torch.bfloat16)
        fz = kda.Fusion(l2norm_qk=True, beta_sigmoid=True, out_gate=gate)
        kda.kda_decode_multi_ex(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), S, d.state_indices,
                                fusion=fz, o=o, S_steps=st)
    else:
        kda.kda_decode_multi(tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta), S, d.state_indices, o=o,
                             S_steps=st)
    torch.cuda.synchronize()
    assert _intact(S_buf, 9.0) and _intact(o_buf, 7.0) and _intact(st_buf, 5.0)


def test_snapshots_write_inside_their_buffer():
    p = synth.prefill_inputs([300, 130, 64], 2, s0_std=0.02, seed=903, device="cuda")
    seq = torch.tensor([0, 0, 1, 1, 2], dtype=torch.int32, device="cuda")
    pos = torch.tensor([64, 300, 128, 130, 64], dtype=torch.int32, device="cuda")
    ss_buf, ss = _padded((5, 2, 128, 128), torch.float32, 3.0)
    kda.kda_prefill_snapshots(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, seq, pos, p.S0, S_snap=ss)
    torch.cuda.synchronize()
    assert _intact(ss_buf, 3.0)


def test_backward_writes_inside_its_buffers():
    p = synth.prefill_inputs([200, 77, 1], 3, s0_std=0.02, seed=904, device="cuda")
    T, H = p.q.shape[:2]
    N = len(p.lengths)
    dO = torch.randn(p.q.shape, device="cuda").to(p.q.dtype)
    dSf = torch.randn((N, H, 128, 128), device="cuda") * 0.1
    shapes = [(T, H, 128)] * 4 + [(T, H), (N, H, 128, 128)]
    bufs = [_padded(s, torch.float32, 11.0) for s in shapes]
    kda.kda_prefill_backward(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, dO, p.S0, dSf,
                             grads=tuple(b[1] for b in bufs))
    torch.cuda.synchronize()
    for buf, _ in bufs:
        assert _intact(buf, 11.0)
