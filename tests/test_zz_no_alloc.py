"""kda_prefill_noalloc: prefill for callers that cannot allocate device memory.

Such a caller (a plugin that an engine hands only its own tensors after the
engine reserved all of HBM, or a path where cudaMalloc's implicit device
synchronisation is not allowed) cannot pass a workspace; this entry point
uses a fixed scratch array inside libkda instead.  The test calls it through
the C ABI on three batches in a row: two too large for the array to hold
the two-pass operand images (the single-pass kernel runs) and one small
enough that it does (the two-pass kernels run, with their chunk table in the
array).  Each result is checked against kda_prefill's on the same inputs and
against the fp64 oracle.  This file is collected last so a run that stops at
the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import synth
from tests.conftest import cuda_ok
from tests.gpu_util import TOL, host, oracle_prefill_heads, rell2

pytestmark = [pytest.mark.gpu, pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")]


def _noalloc_fn():
    lib = kda.load_library()
    fn = lib.kda_prefill_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, P, P, ctypes.c_int, P, P, P, P, i32, i64, i32, i32, i32, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


NOALLOC_SCRATCH_BYTES = 4 * 65536  # the library's fixed array: 65,536 int32


def _two_pass_fits(p) -> bool:
    T, H, _ = p.q.shape
    return kda.kda_prefill_workspace_bytes(torch.bfloat16, len(p.lengths), T, H) <= NOALLOC_SCRATCH_BYTES


def test_noalloc_prefill_matches_prefill_and_oracle():
    fn = _noalloc_fn()
    batches = [synth.prefill_inputs([300, 0, 77, 1000, 64], 4, s0_std=0.02, seed=501, device="cuda"),
               synth.prefill_inputs([129, 5], 3, s0_std=0.02, seed=502, device="cuda"),
               synth.prefill_inputs([64], 1, s0_std=0.02, seed=504, device="cuda")]
    assert [_two_pass_fits(p) for p in batches] == [False, False, True]
    for p in batches:
        o_ref, sf_ref = kda.kda_prefill(p.q, p.k, p.v, p.log_alpha, p.beta, p.cu_seqlens, p.S0)
        o = torch.empty_like(p.q)
        sf = torch.empty_like(sf_ref)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        T, H, _ = p.q.shape
        st = fn(_ptr(p.q), _ptr(p.k), _ptr(p.v), kda.KDA_DTYPE_BF16, _ptr(p.log_alpha), _ptr(p.beta),
                _ptr(p.S0), _ptr(p.cu_seqlens), len(p.lengths), T, H, 128, 128, _ptr(o), _ptr(sf),
                _ptr(status), _stream())
        assert st == kda.KDA_OK, kda.kda_status_string(st)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert rell2(host(o), host(o_ref)) < TOL
        assert rell2(host(sf), host(sf_ref)) < TOL
        cu = p.cu_seqlens.cpu().tolist()
        for n, (_, o_or, sf_or) in enumerate(oracle_prefill_heads(p)):
            if cu[n + 1] > cu[n]:
                assert rell2(host(o[cu[n]:cu[n + 1]]), o_or) < TOL, n
            assert rell2(host(sf[n]), sf_or) < TOL, n


def test_noalloc_rejects_what_its_scratch_cannot_hold():
    fn = _noalloc_fn()
    p = synth.prefill_inputs([10], 1, seed=503, device="cuda")
    o = torch.empty_like(p.q)
    sf = torch.empty((1, 1, 128, 128), dtype=torch.float32, device="cuda")
    too_many = 65536 + 1
    st = fn(_ptr(p.q), _ptr(p.k), _ptr(p.v), kda.KDA_DTYPE_BF16, _ptr(p.log_alpha), _ptr(p.beta), None,
            _ptr(p.cu_seqlens), too_many, 10, 1, 128, 128, _ptr(o), _ptr(sf), None, _stream())
    assert st == kda.KDA_ERR_WORKSPACE
    st = fn(_ptr(p.q), _ptr(p.k), _ptr(p.v), kda.KDA_DTYPE_F32, _ptr(p.log_alpha), _ptr(p.beta), None,
            _ptr(p.cu_seqlens), 1, 10, 1, 128, 128, _ptr(o), _ptr(sf), None, _stream())
    assert st == kda.KDA_ERR_UNSUPPORTED
