"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments with a status code before any
CUDA call (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

import chunked_delta_rule_kla_gb300 as kla
from chunked_delta_rule_kla_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kla.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kla.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KLA_API\s+[\w\s\*]*?\b(kla_\w+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(kla.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    names = {0: "KLA_OK", 1: "KLA_ERR_INVALID_ARG", 2: "KLA_ERR_UNSUPPORTED",
             3: "KLA_ERR_WORKSPACE", 4: "KLA_ERR_CUDA", 5: "KLA_ERR_DEVICE_TIMEOUT"}
    for code, name in names.items():
        assert kla.kla_status_string(code) == name
    assert kla.kla_status_string(99) == "KLA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    n = lib.kla_chunk_fwd_workspace_bytes(8, 4096, 8, 128, 128, 64, kla.KLA_IO_BF16)
    assert n >= 256 and n % 256 == 0
    assert lib.kla_chunk_fwd_workspace_bytes(1, 1, 1, 128, 128, 64, kla.KLA_IO_FP32) >= 256
    assert lib.kla_chunk_fwd_workspace_bytes(1, 0, 1, 64, 64, 64, kla.KLA_IO_FP32) >= 256
    assert lib.kla_chunk_fwd_workspace_bytes(1, 16, 1, 96, 128, 64, 0) == 0   # dk unsupported
    assert lib.kla_chunk_fwd_workspace_bytes(1, 16, 1, 128, 128, 32, 0) == 0  # chunk unsupported
    assert lib.kla_chunk_fwd_workspace_bytes(-1, 16, 1, 128, 128, 64, 0) == 0
    assert lib.kla_chunk_fwd_workspace_bytes(1, 16, 1, 128, 128, 64, 7) == 0  # bad io enum


# Fake, 256-byte aligned, never dereferenced "device" addresses: every call
# below must fail validation before touching them.
P = 0x10000000
WS = 0x20000000


def _fwd(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, eta=P, eps=1e-6, h0=None, o=P, hT=None, B=1, T=64, H=1,
             dk=128, dv=128, chunk=64, io=kla.KLA_IO_BF16, ws=WS, wsb=256, stream=None)
    a.update(kw)
    return lib.kla_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["eta"], a["eps"], a["h0"], a["o"],
                             a["hT"], a["B"], a["T"], a["H"], a["dk"], a["dv"], a["chunk"],
                             a["io"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), kla.KLA_ERR_INVALID_ARG),
    (dict(k=None), kla.KLA_ERR_INVALID_ARG),
    (dict(v=None), kla.KLA_ERR_INVALID_ARG),
    (dict(g=None), kla.KLA_ERR_INVALID_ARG),
    (dict(eta=None), kla.KLA_ERR_INVALID_ARG),
    (dict(o=None), kla.KLA_ERR_INVALID_ARG),
    (dict(B=-1), kla.KLA_ERR_INVALID_ARG),
    (dict(T=-5), kla.KLA_ERR_INVALID_ARG),
    (dict(io=3), kla.KLA_ERR_INVALID_ARG),
    (dict(eps=-1.0), kla.KLA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), kla.KLA_ERR_INVALID_ARG),
    (dict(q=P + 4), kla.KLA_ERR_INVALID_ARG),            # misaligned
    (dict(g=P + 2), kla.KLA_ERR_INVALID_ARG),
    (dict(dk=96), kla.KLA_ERR_UNSUPPORTED),
    (dict(dv=256), kla.KLA_ERR_UNSUPPORTED),
    (dict(chunk=32), kla.KLA_ERR_UNSUPPORTED),
    (dict(H=70000), kla.KLA_ERR_UNSUPPORTED),
    (dict(ws=None), kla.KLA_ERR_WORKSPACE),
    (dict(wsb=128), kla.KLA_ERR_WORKSPACE),
    (dict(ws=WS + 16), kla.KLA_ERR_WORKSPACE),
])
def test_chunk_fwd_rejects(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _dec(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, eta=P, eps=1e-6, S=P, o=P, B=2, H=2, dk=128, dv=128,
             io=kla.KLA_IO_BF16, stream=None)
    a.update(kw)
    return lib.kla_decode_step(a["q"], a["k"], a["v"], a["g"], a["eta"], a["eps"], a["S"],
                               a["o"], a["B"], a["H"], a["dk"], a["dv"], a["io"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(S=None), kla.KLA_ERR_INVALID_ARG),
    (dict(o=None), kla.KLA_ERR_INVALID_ARG),
    (dict(q=None), kla.KLA_ERR_INVALID_ARG),
    (dict(H=-1), kla.KLA_ERR_INVALID_ARG),
    (dict(io=9), kla.KLA_ERR_INVALID_ARG),
    (dict(S=P + 8), kla.KLA_ERR_INVALID_ARG),
    (dict(eps=-0.5), kla.KLA_ERR_INVALID_ARG),
    (dict(dk=32), kla.KLA_ERR_UNSUPPORTED),
    (dict(dv=100), kla.KLA_ERR_UNSUPPORTED),
])
def test_decode_rejects(lib, kw, code):
    assert _dec(lib, **kw) == code


def test_empty_problems_are_no_ops(lib):
    # B*H == 0: nothing to do, no CUDA call, OK even with null tensors.
    assert _fwd(lib, B=0, q=None, k=None, v=None, g=None, eta=None, o=None) == kla.KLA_OK
    assert _dec(lib, H=0, q=None, k=None, v=None, g=None, eta=None, S=None, o=None) == kla.KLA_OK


def test_workspace_check_rejects_small(lib):
    assert lib.kla_workspace_check(None, 256, None) == kla.KLA_ERR_WORKSPACE
    assert lib.kla_workspace_check(WS, 16, None) == kla.KLA_ERR_WORKSPACE


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import importlib
    mod = importlib.import_module("chunked_delta_rule_kla_gb300")
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        mod.load_library(str(tmp_path / "missing.so"))


# kla_chunk_fwd_noalloc keeps its scratch in a fixed 16 MiB array: a problem
# whose workspace would be larger is refused before any CUDA call.
NOALLOC_MAX = 16 << 20


def _noalloc(lib, B, T, H, dk=128, dv=128):
    return lib.kla_chunk_fwd_noalloc(P, P, P, P, P, ctypes.c_float(1e-6), None, P, None, B, T, H,
                                     dk, dv, 64, kla.KLA_IO_BF16, None)


def _largest_t_under(lib, B, H, limit):
    lo, hi = 64, 64 * 4096
    while hi - lo > 64:
        mid = (lo + hi) // 2 // 64 * 64
        if lib.kla_chunk_fwd_workspace_bytes(B, mid, H, 128, 128, 64, kla.KLA_IO_BF16) <= limit:
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("B,H", [(1, 1), (2, 8), (1, 40)])
def test_noalloc_rejects_beyond_its_array(lib, B, H):
    t_fit = _largest_t_under(lib, B, H, NOALLOC_MAX)
    assert lib.kla_chunk_fwd_workspace_bytes(B, t_fit, H, 128, 128, 64, kla.KLA_IO_BF16) <= NOALLOC_MAX
    t_over = t_fit + 64
    assert lib.kla_chunk_fwd_workspace_bytes(B, t_over, H, 128, 128, 64, kla.KLA_IO_BF16) > NOALLOC_MAX
    assert _noalloc(lib, B, t_over, H) == kla.KLA_ERR_WORKSPACE
    # about 650 records of 25,344 bytes (fewer when the scan's maps share the array)
    assert B * H * t_fit <= 662 * 64


def test_decode_step_checked_rejects(lib):
    args = [P, P, P, P, P, ctypes.c_float(1e-6), P, P, 2, 2, 128, 128, kla.KLA_IO_BF16,
            kla.KLA_BETA_KACZMARZ]
    assert lib.kla_decode_step_checked(*args, WS + 16, None) == kla.KLA_ERR_WORKSPACE   # misaligned record
    bad = list(args)
    bad[13] = 7
    assert lib.kla_decode_step_checked(*bad, WS, None) == kla.KLA_ERR_INVALID_ARG
    bad = list(args)
    bad[6] = None
    assert lib.kla_decode_step_checked(*bad, WS, None) == kla.KLA_ERR_INVALID_ARG


# ---- kla_loglinear_fwd: sizes and argument checks (host side, no launch)

def _ll(lib, **kw):
    a = dict(q=P, k=P, v=P, g=P, eta=P, lam=P, L=None, eps=1e-6, o=P, B=1, T=300, H=2, dk=128, dv=128,
             chunk=64, io=kla.KLA_IO_BF16, beta=kla.KLA_BETA_KACZMARZ, ws=WS, wsb=None, stream=None)
    a.update(kw)
    if a["L"] is None:
        a["L"] = lib.kla_loglinear_num_levels(max(a["T"], 0))
    if a["wsb"] is None:
        a["wsb"] = lib.kla_loglinear_workspace_bytes(a["B"], a["T"], a["H"], 128, 128, 64, kla.KLA_IO_BF16)
    return lib.kla_loglinear_fwd(a["q"], a["k"], a["v"], a["g"], a["eta"], a["lam"], a["L"],
                                 ctypes.c_float(a["eps"]), a["o"], a["B"], a["T"], a["H"], a["dk"], a["dv"],
                                 a["chunk"], a["io"], a["beta"], a["ws"], a["wsb"], a["stream"])


def test_loglinear_levels(lib):
    # 1 + ceil(log2 T): a pair of tokens below T is at most at level ceil(log2 T)
    for T, want in ((1, 1), (2, 2), (3, 3), (64, 7), (65, 8), (128, 8), (129, 9), (4096, 13)):
        assert lib.kla_loglinear_num_levels(T) == want, T


def test_loglinear_workspace_bytes(lib):
    # bf16, d = 128 (the tensor-core path): the error record, one 25,344-byte
    # chunk record per (b, h, chunk) and the fp32 accumulator [B, T, H, 128]
    B, T, H = 2, 300, 3
    n = lib.kla_loglinear_workspace_bytes(B, T, H, 128, 128, 64, kla.KLA_IO_BF16)
    nch = (T + 63) // 64
    want = 256 + B * H * nch * 25344 + 4 * B * T * H * 128
    assert n == (want + 255) // 256 * 256
    assert lib.kla_loglinear_workspace_bytes(B, T, H, 128, 128, 64, kla.KLA_IO_FP32) >= 256
    assert lib.kla_loglinear_workspace_bytes(B, T, H, 64, 128, 64, kla.KLA_IO_BF16) >= 256
    assert lib.kla_loglinear_workspace_bytes(B, T, H, 96, 128, 64, kla.KLA_IO_BF16) == 0
    assert lib.kla_loglinear_workspace_bytes(B, T, H, 128, 128, 32, kla.KLA_IO_BF16) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), kla.KLA_ERR_INVALID_ARG),
    (dict(lam=None), kla.KLA_ERR_INVALID_ARG),
    (dict(o=None), kla.KLA_ERR_INVALID_ARG),
    (dict(L=8), kla.KLA_ERR_INVALID_ARG),             # T = 300 needs 10 levels
    (dict(eps=-1.0), kla.KLA_ERR_INVALID_ARG),
    (dict(beta=7), kla.KLA_ERR_INVALID_ARG),
    (dict(q=P + 8), kla.KLA_ERR_INVALID_ARG),          # not 16-byte aligned
    (dict(lam=P + 2), kla.KLA_ERR_INVALID_ARG),        # not 4-byte aligned
    (dict(dk=96), kla.KLA_ERR_UNSUPPORTED),
    (dict(chunk=32), kla.KLA_ERR_UNSUPPORTED),
    (dict(ws=None), kla.KLA_ERR_WORKSPACE),
    (dict(ws=WS + 16), kla.KLA_ERR_WORKSPACE),         # not 256-byte aligned
    (dict(wsb=256), kla.KLA_ERR_WORKSPACE),            # too small
])
def test_loglinear_fwd_rejects(lib, kw, code):
    assert _ll(lib, **kw) == code


def test_loglinear_fwd_empty_problem_is_a_no_op(lib):
    # no tokens: nothing to compute, the pointers and the workspace are not read
    assert _ll(lib, T=0, q=None, ws=None, wsb=0) == kla.KLA_OK
    assert _ll(lib, B=0, q=None, ws=None, wsb=0) == kla.KLA_OK


# ---- kla_deltakata_fwd: sizes and argument checks (host side, no launch)

def _dk_ws_want(B, T, H):
    nch = (T + 63) // 64
    flags = 0
    if 2 * B * H <= 152:   # the fused grid's role counters and ready flags
        flags = (4 * (2 + B * H * nch) + 255) // 256 * 256
    return 256 + B * H * nch * 58112 + flags


@pytest.mark.parametrize("B,T,H", [(1, 300, 2), (8, 4096, 8), (1, 2100, 40), (1, 128, 140)])
def test_deltakata_workspace_bytes(lib, B, T, H):
    # the error record, one 58,112-byte record per (b, h, chunk) (the prefill's
    # 25,344 bytes and two 16 KB feature tiles), then the fused grid's flags
    assert lib.kla_deltakata_fwd_workspace_bytes(B, T, H, 15, 128, 64, kla.KLA_IO_BF16) == _dk_ws_want(B, T, H)


@pytest.mark.parametrize("B,T,H", [(1, 4096, 2), (1, 131072, 16), (1, 4096, 100), (2, 300, 70)])
def test_deltakata_workspace_is_the_prefills_with_larger_records(lib, B, T, H):
    # the chunk-level scan, chunk ranges and the prep-then-carry shapes: the
    # prefill's workspace with each record grown by the two feature tiles
    nch = (T + 63) // 64
    plain = lib.kla_chunk_fwd_workspace_bytes(B, T, H, 128, 128, 64, kla.KLA_IO_BF16)
    fused = lib.kla_deltakata_fwd_workspace_bytes(B, T, H, 15, 128, 64, kla.KLA_IO_BF16)
    assert fused - plain == B * H * nch * (58112 - 25344)


@pytest.mark.parametrize("args", [
    (1, 300, 2, 16, 128, 64, kla.KLA_IO_BF16),     # p(p+1)/2 > 128
    (1, 300, 2, 0, 128, 64, kla.KLA_IO_BF16),
    (1, 300, 2, 15, 64, 64, kla.KLA_IO_BF16),      # d_v = 64
    (1, 300, 2, 15, 128, 32, kla.KLA_IO_BF16),
    (1, 300, 2, 15, 128, 64, kla.KLA_IO_FP32),
])
def test_deltakata_workspace_bytes_unsupported(lib, args):
    assert lib.kla_deltakata_fwd_workspace_bytes(*args) == 0


def _dkf(lib, **kw):
    a = dict(xq=P, xk=P, v=P, g=P, eta=P, eps=1e-6, h0=None, o=P, hT=None, B=1, T=300, H=2, p=15,
             dv=128, chunk=64, io=kla.KLA_IO_BF16, beta=kla.KLA_BETA_KACZMARZ, ws=WS, wsb=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = _dk_ws_want(a["B"], a["T"], a["H"])
    return lib.kla_deltakata_fwd(a["xq"], a["xk"], a["v"], a["g"], a["eta"], ctypes.c_float(a["eps"]),
                                 a["h0"], a["o"], a["hT"], a["B"], a["T"], a["H"], a["p"], a["dv"],
                                 a["chunk"], a["io"], a["beta"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(xq=None), kla.KLA_ERR_INVALID_ARG),
    (dict(xk=None), kla.KLA_ERR_INVALID_ARG),
    (dict(v=None), kla.KLA_ERR_INVALID_ARG),
    (dict(xq=P + 2), kla.KLA_ERR_INVALID_ARG),        # not 4-byte aligned
    (dict(v=P + 4), kla.KLA_ERR_INVALID_ARG),         # not 16-byte aligned
    (dict(eps=-1.0), kla.KLA_ERR_INVALID_ARG),
    (dict(beta=5), kla.KLA_ERR_INVALID_ARG),
    (dict(p=0), kla.KLA_ERR_INVALID_ARG),
    (dict(p=16), kla.KLA_ERR_UNSUPPORTED),
    (dict(dv=64), kla.KLA_ERR_UNSUPPORTED),
    (dict(io=kla.KLA_IO_FP32), kla.KLA_ERR_UNSUPPORTED),
    (dict(ws=None), kla.KLA_ERR_WORKSPACE),
    (dict(ws=WS + 64), kla.KLA_ERR_WORKSPACE),
    (dict(wsb=4096), kla.KLA_ERR_WORKSPACE),
])
def test_deltakata_fwd_rejects(lib, kw, code):
    assert _dkf(lib, **kw) == code


def test_deltakata_fwd_no_heads_is_a_no_op(lib):
    assert _dkf(lib, B=0, xq=None, xk=None, v=None, g=None, eta=None, o=None, wsb=256) == kla.KLA_OK


@pytest.mark.parametrize("B,T,H", [(0, 300, 2), (2, 300, 0), (2, 0, 3)])
def test_segment_policy_and_workspace_of_empty_problems(lib, B, T, H):
    # no heads or no tokens: one segment, and a workspace of the error record
    # plus whatever the path keeps per chunk (nothing here)
    assert lib.kla_chunk_fwd_auto_segments(B, T, H, 128, 128, 64, kla.KLA_IO_BF16) == 1
    assert lib.kla_chunk_fwd_auto_segments(B, T, H, 64, 64, 64, kla.KLA_IO_BF16) == 1
    assert lib.kla_chunk_fwd_workspace_bytes(B, T, H, 128, 128, 64, kla.KLA_IO_BF16) >= 256
    assert lib.kla_deltakata_fwd_workspace_bytes(B, T, H, 15, 128, 64, kla.KLA_IO_BF16) >= 256
