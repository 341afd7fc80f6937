"""The prefill kernels' wind-down after an expired on-chip wait, exercised without a fault.

Every on-chip wait of the prefill kernels is bounded.  When a pipeline wait (for a copy or a
tensor-core product the next step needs) expires, the kernel sets KDA_DEV_TIMEOUT, waits for that
same operation again with a separate drain limit before anything reuses its buffers, stops its
loop, waits for every copy and product of its own still in flight, releases TMEM and returns.

A second copy of the library built with KDA_PIPE_WAIT_CYCLES=0 makes every pipeline wait that is
not already complete on its first poll expire; the drain waits keep their normal limit.  Nothing
stalls on purpose: every awaited copy and product completes as usual.  Each test calls that copy
through the C ABI, checks that the call returns and the status word carries KDA_DEV_TIMEOUT, then
runs the normal library in the same process and checks its result against the fp64 oracle.
"""
import ctypes
import os

import pytest
import torch

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import _binding, _build, synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, oracle_prefill_heads, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]

WAIT_DIR = os.path.join(_build.BUILD_DIR, "pipe_wait_0")


@pytest.fixture(scope="module")
def wait_lib():
    path = _build.build(extra_flags=["-DKDA_PIPE_WAIT_CYCLES=0"], lib_path=os.path.join(WAIT_DIR, "libkda_pipe_wait_0.so"),
                        build_dir=WAIT_DIR)
    return _binding.load_library(path)  # its own handle: the normal library stays the package's


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(lib, p, path, fusion=None):
    T, H, _ = p.q.shape
    N = len(p.lengths)
    o = torch.full_like(p.q, 7.0)
    sf = torch.full((N, H, 128, 128), 7.0, dtype=torch.float32, device="cuda")
    wsb = (kda.kda_prefill_workspace_bytes if path == "two_pass" else kda.kda_prefill_min_workspace_bytes)(
        p.q.dtype, N, T, H)
    work = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (_ptr(p.q), _ptr(p.k), _ptr(p.v), kda.KDA_DTYPE_BF16, _ptr(p.log_alpha), _ptr(p.beta), _ptr(p.S0),
            _ptr(p.cu_seqlens), N, T, H, 128, 128, _ptr(o), _ptr(sf))
    if fusion is None:
        rc = lib.kda_prefill(*args, _ptr(work), work.numel(), _ptr(status), stream)
    else:
        fz = fusion.c_struct()
        rc = lib.kda_prefill_ex(*args, ctypes.byref(fz), _ptr(work), work.numel(), _ptr(status), stream)
    torch.cuda.synchronize()
    return rc, int(status.item())


def _check_normal_call(p):
    o, sf = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
    torch.cuda.synchronize()
    cu = p.cu_seqlens.cpu().tolist()
    for n, (_, o_ref, sf_ref) in enumerate(oracle_prefill_heads(p)):
        assert rell2(host(o[cu[n]:cu[n + 1]]), o_ref) < TOL
        assert rell2(host(sf[n]), sf_ref) < TOL


@pytest.mark.parametrize("path", ["two_pass", "single_pass"])
def test_expired_waits_report_timeout_and_the_next_call_is_exact(wait_lib, path):
    p = synth.prefill_inputs([300, 77, 130], 3, s0_std=0.02, seed=811, device="cuda")
    rc, status = _call(wait_lib, p, path)
    assert rc == kda.KDA_OK
    assert status & kda.KDA_DEV_TIMEOUT
    _check_normal_call(p)


def test_expired_waits_in_the_one_set_scan(wait_lib):
    """A scan grid larger than the SM count runs with one operand set per CTA (two CTAs per SM), whose
    next chunk's copies are issued at the end of each step: its expired waits wind down the same way."""
    lengths = [300, 77, 130, 0, 64, 65, 1, 200, 129, 63, 500, 7]
    H = torch.cuda.get_device_properties(0).multi_processor_count // (2 * len(lengths)) + 1
    p = synth.prefill_inputs(lengths, H, s0_std=0.02, seed=814, device="cuda")
    rc, status = _call(wait_lib, p, "two_pass")
    assert rc == kda.KDA_OK
    assert status & kda.KDA_DEV_TIMEOUT
    _check_normal_call(p)


def test_expired_waits_with_the_output_gate(wait_lib):
    """With the output gate the scan's waits expire the same way, and the gate's pass after the scan
    (which waits on nothing) still runs to the end of the call."""
    p = synth.prefill_inputs([300, 77], 2, s0_std=0.02, seed=812, device="cuda")
    gate = torch.randn(p.q.shape, device="cuda").to(p.q.dtype)
    rc, status = _call(wait_lib, p, "two_pass", kda.Fusion(out_gate=gate))
    assert rc == kda.KDA_OK
    assert status & kda.KDA_DEV_TIMEOUT
    _check_normal_call(p)


def test_expired_wait_in_the_multi_token_decode(wait_lib):
    """The multi-token decode waits (bounded) for the bulk copy of each unit's state; its first wait
    follows the copy's issue at once, so with the zero limit it expires, the CTA drains that copy and
    returns with KDA_DEV_TIMEOUT.  A normal call afterwards matches the oracle."""
    import numpy as np
    import oracle
    N, H, T = 64, 4, 3
    d = synth.decode_inputs(N, H, T, seed=813, device="cuda")
    tm = lambda x: x.transpose(0, 1).contiguous()
    q, k, v, la, b = tm(d.q), tm(d.k), tm(d.v), tm(d.log_alpha), tm(d.beta)
    S = d.S.clone()
    o = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = wait_lib.kda_decode_multi(_ptr(q), _ptr(k), _ptr(v), kda.KDA_DTYPE_BF16, _ptr(la), _ptr(b), _ptr(S), N,
                                   None, N, T, H, 128, 128, _ptr(o), None, _ptr(status), stream)
    torch.cuda.synchronize()
    assert rc == kda.KDA_OK
    assert int(status.item()) & kda.KDA_DEV_TIMEOUT
    S = d.S.clone()
    S_ref = host(S).astype(np.float64)
    o_ref = np.stack([oracle.kda_decode_step(host(d.q[t]), host(d.k[t]), host(d.v[t]), host(d.log_alpha[t]),
                                             host(d.beta[t]), S_ref, None) for t in range(T)], axis=1)
    o = kda.kda_decode_multi(q, k, v, la, b, S, None)
    torch.cuda.synchronize()
    assert rell2(host(o), o_ref) < TOL
    assert rell2(host(S), S_ref) < 1e-5
