"""CPU-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments synchronously (no kernel runs)."""
import ctypes
import os
import re

import pytest

import linear_attention_chunkwise_gb300 as kda
from linear_attention_chunkwise_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kda.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]*?\b(kda_\w+)\s*\(", src)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(kda.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.kda_abi_version() == 1
    assert kda.kda_status_string(kda.KDA_OK) == "KDA_OK"
    assert kda.kda_status_string(kda.KDA_ERR_WORKSPACE) == "KDA_ERR_WORKSPACE"
    assert kda.kda_status_string(99) == "KDA_ERR_UNKNOWN"


BLOB = 67072  # bytes of prepared operands per (chunk, head), two-pass path


def test_workspace_bytes(lib):
    # single-pass path: schedule (+ bf16 copies of fp32 inputs)
    assert kda.kda_prefill_min_workspace_bytes(kda.KDA_DTYPE_BF16, 16, 1000, 32) == 256
    assert kda.kda_prefill_min_workspace_bytes(kda.KDA_DTYPE_F32, 1, 256, 2) == 256 + 3 * 256 * 2 * 128 * 2
    # two-pass path: schedule + chunk table + (copies) + (ceil(T/64) + N) chunks x H operand images, then
    # (256-byte aligned) one fp32 state per (sequence, head) carried between scan pieces
    up = lambda x: -(-x // 256) * 256
    STATE = 128 * 128 * 4
    assert kda.kda_prefill_workspace_bytes(kda.KDA_DTYPE_BF16, 16, 1000, 32) == \
        up(256 + 256 + (16 + 16) * 32 * BLOB) + 16 * 32 * STATE
    assert kda.kda_prefill_workspace_bytes(kda.KDA_DTYPE_F32, 1, 256, 2) == \
        up(256 + 256 + 3 * 256 * 2 * 128 * 2 + (4 + 1) * 2 * BLOB) + 2 * STATE
    for fn in (kda.kda_prefill_workspace_bytes, kda.kda_prefill_min_workspace_bytes):
        assert fn(kda.KDA_DTYPE_BF16, -1, 10, 2) == 0
        assert fn(7, 1, 10, 2) == 0
        assert fn(kda.KDA_DTYPE_BF16, 1, 10, 2, 64, 128) == 0


def _fake(addr):
    return ctypes.c_void_p(addr)


BASE = 1 << 40  # fake, never dereferenced: validation fails before any CUDA call


def _prefill(lib, **over):
    T, H, N = 128, 2, 1
    tok = T * H * 128
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, o=BASE + 12 * tok, Sf=BASE + 14 * tok,
             ws=BASE + 20 * tok, wsb=1 << 20, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]), P(a["S0"]),
                           P(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"], P(a["o"]), P(a["Sf"]), P(a["ws"]),
                           a["wsb"], P(a["status"]), None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(dv=256), kda.KDA_ERR_UNSUPPORTED),
    (dict(dtype=5), kda.KDA_ERR_UNSUPPORTED),
    (dict(q=None), kda.KDA_ERR_INVALID_ARG),
    (dict(cu=None), kda.KDA_ERR_INVALID_ARG),
    (dict(q=BASE + 8), kda.KDA_ERR_INVALID_ARG),                 # misaligned
    (dict(ws=BASE + 20 * 128 * 2 * 128 + 16), kda.KDA_ERR_INVALID_ARG),  # workspace not 256-aligned
    (dict(wsb=16), kda.KDA_ERR_WORKSPACE),
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(N=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(o=BASE + 2 * 128 * 2 * 128), kda.KDA_ERR_INVALID_ARG),  # o overlaps k
    (dict(Sf=BASE + 12 * 128 * 2 * 128), kda.KDA_ERR_INVALID_ARG),  # S_final overlaps o
    (dict(S0=BASE + 30 * 128 * 2 * 128, Sf=BASE + 30 * 128 * 2 * 128 + 4096), kda.KDA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_arguments(lib, over, expect):
    assert _prefill(lib, **over) == expect


def _snapshots(lib, **over):
    T, H, N = 128, 2, 1
    tok = T * H * 128
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, o=BASE + 12 * tok, Sf=BASE + 14 * tok,
             sseq=BASE + 16 * tok, spos=BASE + 16 * tok + 256, M=2, Ss=BASE + 60 * tok, ws=BASE + 20 * tok,
             wsb=1 << 20, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill_snapshots(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]),
                                     P(a["S0"]), P(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"], P(a["o"]),
                                     P(a["Sf"]), P(a["sseq"]), P(a["spos"]), a["M"], P(a["Ss"]), P(a["ws"]),
                                     a["wsb"], P(a["status"]), None)


@pytest.mark.parametrize("over,expect", [
    (dict(M=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(sseq=None), kda.KDA_ERR_INVALID_ARG),
    (dict(spos=None), kda.KDA_ERR_INVALID_ARG),
    (dict(Ss=None), kda.KDA_ERR_INVALID_ARG),
    (dict(Ss=BASE + 60 * 128 * 2 * 128 + 8), kda.KDA_ERR_INVALID_ARG),    # misaligned
    (dict(Ss=BASE + 12 * 128 * 2 * 128), kda.KDA_ERR_INVALID_ARG),        # S_snap overlaps o
    (dict(Ss=BASE + 19 * 128 * 2 * 128), kda.KDA_ERR_INVALID_ARG),        # S_snap overlaps the workspace
    (dict(wsb=4096), kda.KDA_ERR_WORKSPACE),                              # single-pass workspace only
    (dict(dk=64), kda.KDA_ERR_UNSUPPORTED),
])
def test_prefill_snapshots_rejects_bad_arguments(lib, over, expect):
    assert _snapshots(lib, **over) == expect


def _prefill_ex(lib, fz, **over):
    T, H, N = 128, 2, 1
    tok = T * H * 128
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, o=BASE + 12 * tok, Sf=BASE + 14 * tok,
             ws=BASE + 20 * tok, wsb=1 << 20, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill_ex(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]), P(a["S0"]),
                              P(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"], P(a["o"]), P(a["Sf"]),
                              ctypes.byref(fz), P(a["ws"]), a["wsb"], P(a["status"]), None)


def _fusion(flags=0, l2_eps=1e-6, rms_eps=1e-6, w=None, g=None):
    from linear_attention_chunkwise_gb300._binding import _KdaFusion
    return _KdaFusion(flags, l2_eps, rms_eps, w, g)


GATE = BASE + 40 * 128 * 2 * 128  # a gate buffer clear of every other fake range


@pytest.mark.parametrize("fz,over,expect", [
    (dict(flags=0x8), {}, kda.KDA_ERR_INVALID_ARG),                                  # unknown flag
    (dict(flags=kda.KDA_FUSE_L2NORM_QK, l2_eps=-1.0), {}, kda.KDA_ERR_INVALID_ARG),   # negative eps
    (dict(flags=kda.KDA_FUSE_OUT_GATE), {}, kda.KDA_ERR_INVALID_ARG),                 # no gate
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GATE + 8), {}, kda.KDA_ERR_INVALID_ARG),     # misaligned gate
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=BASE + 12 * 128 * 2 * 128), {}, kda.KDA_ERR_INVALID_ARG),  # gate = o
    (dict(flags=kda.KDA_FUSE_L2NORM_QK), dict(wsb=4096), kda.KDA_ERR_WORKSPACE),      # single-pass workspace
])
def test_prefill_ex_rejects_bad_fusion(lib, fz, over, expect):
    assert _prefill_ex(lib, _fusion(**fz), **over) == expect


def test_decode_ex_rejects_bad_fusion(lib):
    N, H = 4, 2
    io = N * H * 128
    P = _fake
    fz = _fusion(flags=0x10)
    st = lib.kda_decode_step_ex(P(BASE), P(BASE + 2 * io), P(BASE + 4 * io), 0, P(BASE + 6 * io),
                                P(BASE + 10 * io), P(BASE + 20 * io), N, None, N, H, 128, 128, P(BASE + 12 * io),
                                ctypes.byref(fz), None, None)
    assert st == kda.KDA_ERR_INVALID_ARG
    fz = _fusion(flags=kda.KDA_FUSE_OUT_GATE)  # gate missing
    st = lib.kda_decode_step_ex(P(BASE), P(BASE + 2 * io), P(BASE + 4 * io), 0, P(BASE + 6 * io),
                                P(BASE + 10 * io), P(BASE + 20 * io), N, None, N, H, 128, 128, P(BASE + 12 * io),
                                ctypes.byref(fz), None, None)
    assert st == kda.KDA_ERR_INVALID_ARG


def _decode(lib, **over):
    N, H = 4, 2
    io = N * H * 128
    a = dict(q=BASE, k=BASE + 2 * io, v=BASE + 4 * io, dtype=0, la=BASE + 6 * io, beta=BASE + 10 * io,
             S=BASE + (1 << 30), slots=N, idx=None, N=N, H=H, dk=128, dv=128, o=BASE + 12 * io, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_decode_step(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]), P(a["S"]),
                               a["slots"], P(a["idx"]), a["N"], a["H"], a["dk"], a["dv"], P(a["o"]), P(a["status"]),
                               None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=32), kda.KDA_ERR_UNSUPPORTED),
    (dict(S=None), kda.KDA_ERR_INVALID_ARG),
    (dict(slots=2), kda.KDA_ERR_INVALID_ARG),                    # identity slots need num_slots >= N
    (dict(o=BASE + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(o=BASE + (1 << 30) + 64), kda.KDA_ERR_INVALID_ARG),    # o inside S
    (dict(N=0), kda.KDA_OK),                                      # nothing to do
])
def test_decode_rejects_bad_arguments(lib, over, expect):
    assert _decode(lib, **over) == expect


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        kda.load_library(str(tmp_path / "nope.so"))


def _decode_multi(lib, **over):
    N, T, H = 2, 3, 2
    io = N * T * H * 128
    a = dict(q=BASE, k=BASE + 2 * io, v=BASE + 4 * io, dtype=0, la=BASE + 6 * io, beta=BASE + 10 * io,
             S=BASE + (1 << 30), slots=N, idx=None, N=N, T=T, H=H, dk=128, dv=128, o=BASE + 12 * io, steps=None,
             status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_decode_multi(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]), P(a["S"]),
                                a["slots"], P(a["idx"]), a["N"], a["T"], a["H"], a["dk"], a["dv"], P(a["o"]),
                                P(a["steps"]), P(a["status"]), None)


@pytest.mark.parametrize("over,expect", [
    (dict(dv=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(T=0), kda.KDA_OK),
    (dict(q=None), kda.KDA_ERR_INVALID_ARG),
    (dict(steps=BASE + 8), kda.KDA_ERR_INVALID_ARG),                    # misaligned
    (dict(steps=BASE + (1 << 30) + 4096), kda.KDA_ERR_INVALID_ARG),     # S_steps inside S
    (dict(o=BASE + 2 * 2 * 3 * 2 * 128), kda.KDA_ERR_INVALID_ARG),      # o overlaps k
])
def test_decode_multi_rejects_bad_arguments(lib, over, expect):
    assert _decode_multi(lib, **over) == expect


def test_backward_workspace_bytes(lib):
    # schedule + chunk table, then the larger of the forward's operand images and the backward's
    # per-chunk records (180,736 B per chunk-head), o scratch, snapshot entries, and two states
    # (the state and its adjoint) per chunk slot and head; chunk slots = ceil(T/64) + N
    REC = 180736
    for T, H, N in ((128, 2, 1), (1000, 32, 16)):
        slots = -(-T // 64) + N
        o = max(512 + slots * H * BLOB, 512 + slots * H * REC) if N == 1 else \
            max(256 * ((N * 4 + 255) // 256) + 256 * (((N + 3) * 4 + 255) // 256) + slots * H * BLOB,
                256 * ((N * 4 + 255) // 256) + 256 * (((N + 3) * 4 + 255) // 256) + slots * H * REC)
        o = -(-o // 256) * 256
        ent = -(-(slots * 4) // 256) * 256
        want = o + -(-(T * H * 128 * 2) // 256) * 256 + 2 * ent + 2 * slots * H * 128 * 128 * 4
        assert kda.kda_prefill_backward_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H) == want
    assert kda.kda_prefill_backward_workspace_bytes(kda.KDA_DTYPE_BF16, -1, 10, 2) == 0
    assert kda.kda_prefill_backward_workspace_bytes(kda.KDA_DTYPE_BF16, 1, 10, 2, 64, 128) == 0


def _backward(lib, **over):
    T, H, N = 128, 2, 1
    tok = T * H * 128
    need = kda.kda_prefill_backward_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H)
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, dO=BASE + 12 * tok, dSf=None,
             gq=BASE + 20 * tok, gk=BASE + 24 * tok, gv=BASE + 28 * tok, gla=BASE + 32 * tok, gb=BASE + 36 * tok,
             gs0=BASE + 40 * tok, ws=BASE + 64 * tok, wsb=need, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill_backward(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]),
                                    P(a["S0"]), P(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"], P(a["dO"]),
                                    P(a["dSf"]), P(a["gq"]), P(a["gk"]), P(a["gv"]), P(a["gla"]), P(a["gb"]),
                                    P(a["gs0"]), P(a["ws"]), a["wsb"], P(a["status"]), None)


TOK = 128 * 2 * 128


@pytest.mark.parametrize("over,expect", [
    (dict(dk=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(dtype=5), kda.KDA_ERR_UNSUPPORTED),
    (dict(dO=None), kda.KDA_ERR_INVALID_ARG),
    (dict(gq=None), kda.KDA_ERR_INVALID_ARG),
    (dict(gb=None), kda.KDA_ERR_INVALID_ARG),
    (dict(cu=None), kda.KDA_ERR_INVALID_ARG),
    (dict(gk=BASE + 24 * TOK + 8), kda.KDA_ERR_INVALID_ARG),       # misaligned
    (dict(ws=BASE + 64 * TOK + 16), kda.KDA_ERR_INVALID_ARG),      # workspace not 256-aligned
    (dict(wsb=1 << 20), kda.KDA_ERR_WORKSPACE),
    (dict(gv=BASE + 20 * TOK + 4096), kda.KDA_ERR_INVALID_ARG),    # grad_v overlaps grad_q
    (dict(gla=BASE + 12 * TOK), kda.KDA_ERR_INVALID_ARG),          # grad_log_alpha overlaps grad_o
    (dict(gs0=BASE + 70 * TOK), kda.KDA_ERR_INVALID_ARG),          # grad_S0 inside the workspace
    (dict(gq=BASE), kda.KDA_ERR_INVALID_ARG),                      # grad_q overlaps q
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
])
def test_backward_rejects_bad_arguments(lib, over, expect):
    assert _backward(lib, **over) == expect


def test_backward_ex_workspace_bytes(lib):
    # the plain backward's workspace, then normalised q and k (input dtype), sigmoid beta (fp32) and the
    # two inverse norms (fp32) per (token, head), each region 256-byte aligned
    up = lambda x: -(-x // 256) * 256
    for dt, es in ((kda.KDA_DTYPE_BF16, 2), (kda.KDA_DTYPE_F32, 4)):
        for T, H, N in ((128, 2, 1), (1000, 32, 16), (0, 4, 3)):
            plain = kda.kda_prefill_backward_workspace_bytes(dt, N, T, H)
            want = plain + 2 * up(T * H * 128 * es) + up(T * H * 4) + up(T * H * 8)
            assert kda.kda_prefill_backward_ex_workspace_bytes(dt, N, T, H) == want
    assert kda.kda_prefill_backward_ex_workspace_bytes(kda.KDA_DTYPE_BF16, -1, 10, 2) == 0
    assert kda.kda_prefill_backward_ex_workspace_bytes(kda.KDA_DTYPE_BF16, 1, 10, 2, 128, 64) == 0


def _backward_ex(lib, fz, **over):
    T, H, N = 128, 2, 1
    tok = T * H * 128
    need = kda.kda_prefill_backward_ex_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H)
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, dO=BASE + 12 * tok, dSf=None,
             gq=BASE + 20 * tok, gk=BASE + 24 * tok, gv=BASE + 28 * tok, gla=BASE + 32 * tok, gb=BASE + 36 * tok,
             gs0=BASE + 40 * tok, ws=BASE + 64 * tok, wsb=need, status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill_backward_ex(P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]),
                                       P(a["S0"]), P(a["cu"]), a["N"], a["T"], a["H"], a["dk"], a["dv"],
                                       P(a["dO"]), P(a["dSf"]), P(a["gq"]), P(a["gk"]), P(a["gv"]), P(a["gla"]),
                                       P(a["gb"]), P(a["gs0"]), None if fz is None else ctypes.byref(fz),
                                       P(a["ws"]), a["wsb"], P(a["status"]), None)


PLAIN_BWD_WS = 128 * 2 * 128 * 64  # offset of the workspace in the fake layout above


@pytest.mark.parametrize("fz,over,expect", [
    (dict(flags=0x8), {}, kda.KDA_ERR_INVALID_ARG),                                    # unknown flag
    (dict(flags=kda.KDA_FUSE_L2NORM_QK, l2_eps=-1.0), {}, kda.KDA_ERR_INVALID_ARG),     # negative eps
    (dict(flags=kda.KDA_FUSE_OUT_GATE), {}, kda.KDA_ERR_INVALID_ARG),                   # gate missing
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GATE), {}, kda.KDA_ERR_UNSUPPORTED),           # kda_prefill_backward_gated's
    (dict(flags=kda.KDA_FUSE_L2NORM_QK | kda.KDA_FUSE_BETA_SIGMOID), dict(dk=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(flags=kda.KDA_FUSE_BETA_SIGMOID), dict(gq=BASE + 2 * 128 * 2 * 128), kda.KDA_ERR_INVALID_ARG),  # = k
])
def test_backward_ex_rejects_bad_arguments(lib, fz, over, expect):
    assert _backward_ex(lib, _fusion(**fz), **over) == expect


def test_backward_ex_workspace_covers_the_prologue_copies(lib):
    """The plain figure is too small once a prologue flag is set, and the copies' tail is checked for overlap."""
    N, T, H = 1, 128, 2
    plain = kda.kda_prefill_backward_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H)
    fz = _fusion(flags=kda.KDA_FUSE_L2NORM_QK)
    assert _backward_ex(lib, fz, wsb=plain) == kda.KDA_ERR_WORKSPACE
    in_tail = BASE + PLAIN_BWD_WS + plain  # grad_S0 on the normalised-q copy
    assert _backward_ex(lib, fz, gs0=in_tail) == kda.KDA_ERR_INVALID_ARG
    # without prologue flags the tail is not the call's: the same grad_S0 passes every argument check
    # and the call stops only at the device check (no GPU here)
    for none in (None, _fusion(flags=0)):
        assert _backward_ex(lib, none, gs0=in_tail, wsb=plain) == kda.KDA_ERR_CUDA


def test_backward_gated_workspace_bytes(lib):
    # the _ex workspace rounded up to 256 bytes, then 592 blocks x 128 fp32 partial sums of dL/dweight
    up = lambda x: -(-x // 256) * 256
    for dt in (kda.KDA_DTYPE_BF16, kda.KDA_DTYPE_F32):
        for T, H, N in ((128, 2, 1), (1000, 32, 16), (0, 4, 3)):
            ex = kda.kda_prefill_backward_ex_workspace_bytes(dt, N, T, H)
            assert kda.kda_prefill_backward_gated_workspace_bytes(dt, N, T, H) == up(ex) + 592 * 128 * 4
    assert kda.kda_prefill_backward_gated_workspace_bytes(kda.KDA_DTYPE_BF16, -1, 10, 2) == 0
    assert kda.kda_prefill_backward_gated_workspace_bytes(kda.KDA_DTYPE_BF16, 1, 10, 2, 128, 64) == 0


GTOK = 128 * 2 * 128  # elements per [T, H, 128] tensor of the fake gated layout below


def _backward_gated(lib, fz, **over):
    T, H, N = 128, 2, 1
    tok = GTOK
    need = kda.kda_prefill_backward_gated_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H)
    a = dict(q=BASE, k=BASE + 2 * tok, v=BASE + 4 * tok, dtype=0, la=BASE + 6 * tok, beta=BASE + 10 * tok,
             S0=None, cu=BASE + 11 * tok, N=N, T=T, H=H, dk=128, dv=128, dY=BASE + 12 * tok, dSf=None,
             gq=BASE + 20 * tok, gk=BASE + 24 * tok, gv=BASE + 28 * tok, gla=BASE + 32 * tok, gb=BASE + 36 * tok,
             gs0=BASE + 40 * tok, gg=BASE + 52 * tok, gw=BASE + 58 * tok, ws=BASE + 64 * tok, wsb=need,
             status=None)
    a.update(over)
    P = lambda x: None if x is None else _fake(x)
    return lib.kda_prefill_backward_gated(
        P(a["q"]), P(a["k"]), P(a["v"]), a["dtype"], P(a["la"]), P(a["beta"]), P(a["S0"]), P(a["cu"]), a["N"],
        a["T"], a["H"], a["dk"], a["dv"], P(a["dY"]), P(a["dSf"]), P(a["gq"]), P(a["gk"]), P(a["gv"]), P(a["gla"]),
        P(a["gb"]), P(a["gs0"]), P(a["gg"]), P(a["gw"]), None if fz is None else ctypes.byref(fz), P(a["ws"]),
        a["wsb"], P(a["status"]), None)


GGATE = BASE + 48 * GTOK      # bf16 [T, H, 128]: [48, 50) x GTOK bytes
GWEIGHT = BASE + 60 * GTOK    # fp32 [128]


@pytest.mark.parametrize("fz,over,expect", [
    (None, {}, kda.KDA_ERR_INVALID_ARG),                                                       # no fusion
    (dict(flags=kda.KDA_FUSE_L2NORM_QK), {}, kda.KDA_ERR_INVALID_ARG),                          # no gate flag
    (dict(flags=kda.KDA_FUSE_OUT_GATE), {}, kda.KDA_ERR_INVALID_ARG),                           # gate missing
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE, rms_eps=-1.0), {}, kda.KDA_ERR_INVALID_ARG),    # negative eps
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gg=None), kda.KDA_ERR_INVALID_ARG),       # no grad_out_gate
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gg=BASE + 52 * GTOK + 4), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gg=GGATE), kda.KDA_ERR_INVALID_ARG),      # = out_gate
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gg=BASE + 12 * GTOK), kda.KDA_ERR_INVALID_ARG),  # = grad_y
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE, w=GWEIGHT), dict(gw=GWEIGHT), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gw=BASE + 54 * GTOK), kda.KDA_ERR_INVALID_ARG),  # in dgate
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(gw=BASE + 58 * GTOK + 2), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(dk=64), kda.KDA_ERR_UNSUPPORTED),
    (dict(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE), dict(dtype=5), kda.KDA_ERR_UNSUPPORTED),
])
def test_backward_gated_rejects_bad_arguments(lib, fz, over, expect):
    assert _backward_gated(lib, None if fz is None else _fusion(**fz), **over) == expect


def test_backward_gated_workspace_covers_the_partials(lib):
    """The _ex figure is too small, and the partial sums' tail is checked for overlap; a call that passes
    every argument check stops at the device check (no GPU here)."""
    N, T, H = 1, 128, 2
    ex = kda.kda_prefill_backward_ex_workspace_bytes(kda.KDA_DTYPE_BF16, N, T, H)
    fz = _fusion(flags=kda.KDA_FUSE_OUT_GATE, g=GGATE, w=GWEIGHT)
    assert _backward_gated(lib, fz, wsb=ex) == kda.KDA_ERR_WORKSPACE
    ws = BASE + 64 * GTOK
    assert _backward_gated(lib, fz, gw=ws + -(-ex // 256) * 256 + 4096) == kda.KDA_ERR_INVALID_ARG
    assert _backward_gated(lib, fz) == kda.KDA_ERR_CUDA
    assert _backward_gated(lib, fz, gw=None) == kda.KDA_ERR_CUDA
    fz2 = _fusion(flags=kda.KDA_FUSE_OUT_GATE | kda.KDA_FUSE_L2NORM_QK | kda.KDA_FUSE_BETA_SIGMOID, g=GGATE)
    assert _backward_gated(lib, fz2) == kda.KDA_ERR_CUDA


def test_out_gate_may_be_null_without_tokens(lib):
    """With no (token, head) rows the gate, like every zero-size array, may be NULL: the call passes every
    argument check and stops at the device check (no GPU here); with tokens it is required."""
    fz = _fusion(flags=kda.KDA_FUSE_OUT_GATE)
    empty = dict(T=0, q=None, k=None, v=None, la=None, beta=None, dY=None, gq=None, gk=None, gv=None, gla=None,
                 gb=None, gg=None)
    assert _backward_gated(lib, fz, **empty) == kda.KDA_ERR_CUDA
    assert _backward_gated(lib, fz) == kda.KDA_ERR_INVALID_ARG


def test_header_bit_constants_match_the_binding():
    """Every KDA_DEV_* and KDA_FUSE_* bit the header defines has the same value in the Python binding."""
    src = open(os.path.join(ROOT, "include", "kda.h")).read()
    defs = dict(re.findall(r"#define\s+(KDA_(?:DEV|FUSE)_\w+)\s+(0x[0-9a-fA-F]+)u?", src))
    assert {"KDA_DEV_BAD_CU_SEQLENS", "KDA_DEV_BOUNDS", "KDA_FUSE_OUT_GATE"} <= set(defs)
    for name, val in defs.items():
        assert getattr(kda, name) == int(val, 16), name
