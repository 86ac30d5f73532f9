"""Python binding of libkla (the KLA chunkwise prefill and decode step).

Thin ctypes marshalling over the C ABI in ``include/kla.h``: the functions
below carry the ABI's names and hand device pointers, sizes and the current
CUDA stream to the library; every step of the computation runs in the
library's CUDA kernels.  PyTorch only provides device memory and streams.

The library is loaded on first use from ``_build/libkla.so`` (built by
``__graft_entry__.build()`` or ``python -m chunked_delta_rule_kla_gb300._build``).
If it is missing, every op raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

KLA_OK = 0
KLA_ERR_INVALID_ARG = 1
KLA_ERR_UNSUPPORTED = 2
KLA_ERR_WORKSPACE = 3
KLA_ERR_CUDA = 4
KLA_ERR_DEVICE_TIMEOUT = 5

KLA_IO_BF16 = 0
KLA_IO_FP32 = 1

KLA_BETA_KACZMARZ = 0   # beta_t = eta_t / (||k_t||^2 + eps)
KLA_BETA_DIRECT = 1     # beta_t = eta_t (the learned-scalar rule; DeltaNet with g = 0)

# Every symbol include/kla.h declares (checked by the ABI tests).
EXPORTED_SYMBOLS = (
    "kla_chunk_fwd_workspace_bytes",
    "kla_chunk_fwd",
    "kla_chunk_fwd_scan_workspace_bytes",
    "kla_chunk_fwd_scan",
    "kla_chunk_fwd_auto_segments",
    "kla_chunk_fwd_noalloc",
    "kla_chunk_fwd_noalloc_check",
    "kla_chunk_fwd_ex",
    "kla_decode_step",
    "kla_decode_step_ex",
    "kla_decode_step_checked",
    "kla_chunk_bwd_workspace_bytes",
    "kla_chunk_bwd",
    "kla_psd_features",
    "kla_psd_features_bwd",
    "kla_deltakata_fwd_workspace_bytes",
    "kla_deltakata_fwd",
    "kla_loglinear_num_levels",
    "kla_loglinear_workspace_bytes",
    "kla_loglinear_fwd",
    "kla_loglinear_decode_step",
    "kla_workspace_check",
    "kla_status_string",
)


class KlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {kla_status_string(code)} ({code})")


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libkla.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libkla.so is not built ({p}); run `python -c \"import __graft_entry__ as g; g.build()\"`")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.kla_chunk_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kla_chunk_fwd_workspace_bytes.restype = sz
        lib.kla_chunk_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                      i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_chunk_fwd.restype = i
        lib.kla_chunk_fwd_scan_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        lib.kla_chunk_fwd_scan_workspace_bytes.restype = sz
        lib.kla_chunk_fwd_scan.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                           i, i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_chunk_fwd_scan.restype = i
        lib.kla_chunk_fwd_auto_segments.argtypes = [i, i, i, i, i, i, i]
        lib.kla_chunk_fwd_auto_segments.restype = i
        lib.kla_chunk_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                              i, i, i, i, i, i, i, vp]
        lib.kla_chunk_fwd_noalloc.restype = i
        lib.kla_chunk_fwd_noalloc_check.argtypes = [vp]
        lib.kla_chunk_fwd_noalloc_check.restype = i
        lib.kla_decode_step.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, vp]
        lib.kla_decode_step.restype = i
        lib.kla_chunk_fwd_ex.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                         i, i, i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_chunk_fwd_ex.restype = i
        lib.kla_decode_step_ex.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, vp]
        lib.kla_decode_step_ex.restype = i
        lib.kla_decode_step_checked.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, i, vp, vp]
        lib.kla_decode_step_checked.restype = i
        lib.kla_chunk_bwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kla_chunk_bwd_workspace_bytes.restype = sz
        lib.kla_chunk_bwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp,
                                      i, i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_chunk_bwd.restype = i
        i64 = ctypes.c_int64
        lib.kla_psd_features.argtypes = [vp, vp, i64, i, i, i, vp]
        lib.kla_psd_features.restype = i
        lib.kla_psd_features_bwd.argtypes = [vp, vp, vp, i64, i, i, i, vp]
        lib.kla_psd_features_bwd.restype = i
        lib.kla_deltakata_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kla_deltakata_fwd_workspace_bytes.restype = sz
        lib.kla_deltakata_fwd.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, vp,
                                          i, i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_deltakata_fwd.restype = i
        lib.kla_loglinear_num_levels.argtypes = [i]
        lib.kla_loglinear_num_levels.restype = i
        lib.kla_loglinear_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
        lib.kla_loglinear_workspace_bytes.restype = sz
        lib.kla_loglinear_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, f, vp,
                                          i, i, i, i, i, i, i, i, vp, sz, vp]
        lib.kla_loglinear_fwd.restype = i
        lib.kla_loglinear_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i, f, vp, i, vp,
                                                  i, i, i, i, i, i, vp]
        lib.kla_loglinear_decode_step.restype = i
        lib.kla_workspace_check.argtypes = [vp, sz, vp]
        lib.kla_workspace_check.restype = i
        lib.kla_status_string.argtypes = [i]
        lib.kla_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def kla_status_string(code: int) -> str:
    return load_library().kla_status_string(int(code)).decode()


def _io_of(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KLA_IO_BF16
    if t.dtype == torch.float32:
        return KLA_IO_FP32
    raise TypeError(f"q/k/v/o must be bfloat16 or float32, got {t.dtype}")


def _ptr(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr() or None


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def kla_chunk_fwd_workspace_bytes(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16) -> int:
    return int(load_library().kla_chunk_fwd_workspace_bytes(B, T, H, dk, dv, chunk, io))


def kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16, segments=0) -> int:
    return int(load_library().kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, chunk, io, segments))


def kla_chunk_fwd_auto_segments(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16) -> int:
    return int(load_library().kla_chunk_fwd_auto_segments(B, T, H, dk, dv, chunk, io))


def _check_prefill_args(q, k, v, g, eta, h0, o, hT):
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    for name, t in (("k", k), ("v", v), ("o", o)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype {q.dtype}")
    if q.shape != k.shape or v.shape[:3] != k.shape[:3] or o.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, o")
    if g.shape != (B, T, H) or eta.shape != (B, T, H):
        raise ValueError("g and eta must be [B,T,H]")
    for name, t in (("h0", h0), ("hT", hT)):
        if t is not None and tuple(t.shape) != (B, H, dk, dv):
            raise ValueError(f"{name} must be [B,H,dk,dv]")
    return B, T, H, dk, dv, _io_of(q)


def kla_chunk_fwd(q, k, v, g, eta, eps, h0, o, hT, workspace, chunk=64, stream=None) -> None:
    """Enqueue the chunkwise prefill (see include/kla.h) on ``stream``.

    q, k [B,T,H,dk]; v, o [B,T,H,dv] (bf16 or fp32, same dtype); g, eta
    [B,T,H] fp32; h0, hT [B,H,dk,dv] fp32 or None; workspace a uint8 CUDA
    tensor of at least kla_chunk_fwd_workspace_bytes(...) bytes.
    """
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, h0, o, hT)
    rc = load_library().kla_chunk_fwd(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(o, "o"), _ptr(hT, "hT", torch.float32), B, T, H, dk, dv, int(chunk), io,
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_chunk_fwd")


def kla_chunk_fwd_scan(q, k, v, g, eta, eps, h0, o, hT, workspace, segments, chunk=64,
                       stream=None) -> None:
    """kla_chunk_fwd with the chunk-level scan's segment count given (see
    include/kla.h): 0 = automatic, 1 = no scan.  workspace holds at least
    kla_chunk_fwd_scan_workspace_bytes(..., segments) bytes."""
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, h0, o, hT)
    rc = load_library().kla_chunk_fwd_scan(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(o, "o"), _ptr(hT, "hT", torch.float32), B, T, H, dk, dv, int(chunk), io,
        int(segments), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_chunk_fwd_scan")


def kla_chunk_fwd_ex(q, k, v, g, eta, eps, h0, o, hT, workspace, beta=KLA_BETA_KACZMARZ,
                     segments=0, chunk=64, stream=None) -> None:
    """kla_chunk_fwd_scan with the step size chosen by ``beta`` (KLA_BETA_KACZMARZ or
    KLA_BETA_DIRECT, see include/kla.h)."""
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, h0, o, hT)
    rc = load_library().kla_chunk_fwd_ex(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(o, "o"), _ptr(hT, "hT", torch.float32), B, T, H, dk, dv, int(chunk), io,
        int(beta), int(segments), _ptr(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_chunk_fwd_ex")


def kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16) -> int:
    return int(load_library().kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv, chunk, io))


def kla_chunk_bwd(q, k, v, g, eta, eps, h0, grad_o, grad_hT, grad_q, grad_k, grad_v, grad_g,
                  grad_eta, grad_h0, workspace, beta=KLA_BETA_KACZMARZ, chunk=64,
                  stream=None) -> None:
    """Enqueue the chunkwise backward (see include/kla.h): the gradients of
    (o, hT) with respect to q, k, v, g, eta and h0.  grad_q, grad_k, grad_v have
    the I/O dtype of q; grad_g, grad_eta, grad_h0 are fp32; grad_hT and grad_h0
    may be None."""
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, h0, grad_o, grad_hT)
    for name, t, ref in (("grad_q", grad_q, q), ("grad_k", grad_k, k), ("grad_v", grad_v, v)):
        if t.shape != ref.shape or t.dtype != ref.dtype:
            raise ValueError(f"{name} must match the shape and dtype of its input")
    if grad_g.shape != g.shape or grad_eta.shape != eta.shape:
        raise ValueError("grad_g and grad_eta must be [B,T,H]")
    if grad_h0 is not None and tuple(grad_h0.shape) != (B, H, dk, dv):
        raise ValueError("grad_h0 must be [B,H,dk,dv]")
    rc = load_library().kla_chunk_bwd(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(grad_o, "grad_o"), _ptr(grad_hT, "grad_hT", torch.float32),
        _ptr(grad_q, "grad_q"), _ptr(grad_k, "grad_k"), _ptr(grad_v, "grad_v"),
        _ptr(grad_g, "grad_g", torch.float32), _ptr(grad_eta, "grad_eta", torch.float32),
        _ptr(grad_h0, "grad_h0", torch.float32), B, T, H, dk, dv, int(chunk), io, int(beta),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_chunk_bwd")


def kla_psd_features(x, y, stream=None) -> None:
    """DeltaKATA features (see include/kla.h): x [..., p] -> y [..., d_out], same dtype."""
    p, d_out = x.shape[-1], y.shape[-1]
    if y.shape[:-1] != x.shape[:-1] or y.dtype != x.dtype:
        raise ValueError("y must be [..., d_out] with x's leading shape and dtype")
    rows = x.numel() // p if p else 0
    rc = load_library().kla_psd_features(_ptr(x, "x"), _ptr(y, "y"), rows, p, d_out, _io_of(x),
                                         _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_psd_features")


def kla_psd_features_bwd(x, grad_y, grad_x, stream=None) -> None:
    """The derivative of kla_psd_features: grad_y [..., d_out] -> grad_x [..., p]."""
    p, d_out = x.shape[-1], grad_y.shape[-1]
    if grad_x.shape != x.shape or grad_y.shape[:-1] != x.shape[:-1]:
        raise ValueError("shape mismatch among x, grad_y, grad_x")
    for name, t in (("grad_y", grad_y), ("grad_x", grad_x)):
        if t.dtype != x.dtype:
            raise TypeError(f"{name} must have x's dtype")
    rows = x.numel() // p if p else 0
    rc = load_library().kla_psd_features_bwd(_ptr(x, "x"), _ptr(grad_y, "grad_y"),
                                             _ptr(grad_x, "grad_x"), rows, p, d_out, _io_of(x),
                                             _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_psd_features_bwd")


def kla_deltakata_fwd_workspace_bytes(B, T, H, p, dv, chunk=64, io=KLA_IO_BF16) -> int:
    """Workspace of kla_deltakata_fwd; 0 where that shape is not supported."""
    return int(load_library().kla_deltakata_fwd_workspace_bytes(B, T, H, p, dv, chunk, io))


def kla_deltakata_fwd(xq, xk, v, g, eta, eps, h0, o, hT, workspace, beta=KLA_BETA_KACZMARZ,
                      chunk=64, stream=None) -> None:
    """Enqueue DeltaKATA's forward with the features formed inside (see
    include/kla.h): xq, xk [B,T,H,p] bf16; v, o [B,T,H,128] bf16; g, eta
    [B,T,H] fp32; h0, hT [B,H,128,128] fp32 or None."""
    B, T, H, p = xk.shape
    dv = v.shape[-1]
    for name, t in (("xk", xk), ("v", v), ("o", o)):
        if t.dtype != xq.dtype:
            raise TypeError(f"{name} must have xq's dtype {xq.dtype}")
    if xq.shape != xk.shape or v.shape[:3] != xk.shape[:3] or o.shape != v.shape:
        raise ValueError("shape mismatch among xq, xk, v, o")
    if g.shape != (B, T, H) or eta.shape != (B, T, H):
        raise ValueError("g and eta must be [B,T,H]")
    for name, t in (("h0", h0), ("hT", hT)):
        if t is not None and tuple(t.shape) != (B, H, 128, dv):
            raise ValueError(f"{name} must be [B,H,128,dv]")
    rc = load_library().kla_deltakata_fwd(
        _ptr(xq, "xq"), _ptr(xk, "xk"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(o, "o"), _ptr(hT, "hT", torch.float32), B, T, H, p, dv, int(chunk), _io_of(xq),
        int(beta), _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_deltakata_fwd")


def kla_loglinear_num_levels(T) -> int:
    return int(load_library().kla_loglinear_num_levels(int(T)))


def kla_loglinear_workspace_bytes(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16) -> int:
    return int(load_library().kla_loglinear_workspace_bytes(B, T, H, dk, dv, chunk, io))


def kla_loglinear_fwd(q, k, v, g, eta, lam, eps, o, workspace, beta=KLA_BETA_KACZMARZ, chunk=64,
                      stream=None) -> None:
    """Enqueue the Log-Linear gated delta rule (see include/kla.h): lam is
    [B,T,H,L] fp32 with L >= kla_loglinear_num_levels(T); the state starts at zero."""
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, None, o, None)
    if lam.dim() != 4 or tuple(lam.shape[:3]) != (B, T, H):
        raise ValueError("lam must be [B,T,H,L]")
    rc = load_library().kla_loglinear_fwd(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), _ptr(lam, "lam", torch.float32), int(lam.shape[3]),
        float(eps), _ptr(o, "o"), B, T, H, dk, dv, int(chunk), io, int(beta),
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_loglinear_fwd")


def kla_loglinear_decode_step(q, k, v, g, eta, lam, eps, states, t, o, beta=KLA_BETA_KACZMARZ,
                              stream=None) -> None:
    """One Log-Linear decode step for token ``t`` (see include/kla.h): states
    [B,H,L,dk,dv] fp32 (zero-filled before t = 0) are updated in place."""
    B, H, dk = k.shape
    dv = v.shape[-1]
    if tuple(states.shape[:2]) != (B, H) or tuple(states.shape[3:]) != (dk, dv) or lam.shape != states.shape[:3]:
        raise ValueError("states must be [B,H,L,dk,dv] and lam [B,H,L]")
    rc = load_library().kla_loglinear_decode_step(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), _ptr(lam, "lam", torch.float32), int(lam.shape[2]),
        float(eps), _ptr(states, "states", torch.float32), int(t), _ptr(o, "o"), B, H, dk, dv,
        _io_of(q), int(beta), _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_loglinear_decode_step")


def kla_chunk_fwd_noalloc(q, k, v, g, eta, eps, h0, o, hT, chunk=64, stream=None) -> None:
    """kla_chunk_fwd without a workspace, for callers that must not allocate
    device memory: the scratch is an array built into the library (see
    include/kla.h).  Allocates nothing; outputs are the caller's tensors."""
    B, T, H, dk, dv, io = _check_prefill_args(q, k, v, g, eta, h0, o, hT)
    rc = load_library().kla_chunk_fwd_noalloc(
        _ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
        _ptr(eta, "eta", torch.float32), float(eps), _ptr(h0, "h0", torch.float32),
        _ptr(o, "o"), _ptr(hT, "hT", torch.float32), B, T, H, dk, dv, int(chunk), io,
        _stream(stream))
    if rc != KLA_OK:
        raise KlaError(rc, "kla_chunk_fwd_noalloc")


def kla_chunk_fwd_noalloc_check(stream=None) -> int:
    """Synchronise and read the device error record of the last
    kla_chunk_fwd_noalloc call on the current device (status code)."""
    return int(load_library().kla_chunk_fwd_noalloc_check(_stream(stream)))


def kla_decode_step(q, k, v, g, eta, eps, S, o, stream=None, beta=KLA_BETA_KACZMARZ,
                    status=None) -> None:
    """Enqueue one decode step (see include/kla.h); S [B,H,dk,dv] is updated in place.

    q, k [B,H,dk]; v, o [B,H,dv] (bf16 or fp32); g, eta [B,H] fp32.  A ``beta``
    other than KLA_BETA_KACZMARZ goes through kla_decode_step_ex; a ``status``
    tensor (>= 256 bytes on the device, cleared by the caller) through
    kla_decode_step_checked, read back with kla_workspace_check(status).
    """
    B, H, dk = k.shape
    dv = v.shape[-1]
    io = _io_of(q)
    for name, t in (("k", k), ("v", v), ("o", o)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype {q.dtype}")
    if q.shape != k.shape or v.shape[:2] != k.shape[:2] or o.shape != v.shape:
        raise ValueError("shape mismatch among q, k, v, o")
    if g.shape != (B, H) or eta.shape != (B, H) or tuple(S.shape) != (B, H, dk, dv):
        raise ValueError("g, eta must be [B,H] and S [B,H,dk,dv]")
    args = (_ptr(q, "q"), _ptr(k, "k"), _ptr(v, "v"), _ptr(g, "g", torch.float32),
            _ptr(eta, "eta", torch.float32), float(eps), _ptr(S, "S", torch.float32),
            _ptr(o, "o"), B, H, dk, dv, io)
    if status is not None:
        if status.numel() * status.element_size() < 256:
            raise ValueError("status must hold at least 256 bytes")
        rc, name = (load_library().kla_decode_step_checked(*args, int(beta), _ptr(status, "status"),
                                                            _stream(stream)), "kla_decode_step_checked")
    elif beta == KLA_BETA_KACZMARZ:
        rc, name = load_library().kla_decode_step(*args, _stream(stream)), "kla_decode_step"
    else:
        rc, name = load_library().kla_decode_step_ex(*args, int(beta), _stream(stream)), "kla_decode_step_ex"
    if rc != KLA_OK:
        raise KlaError(rc, name)


def kla_workspace_check(workspace, stream=None) -> int:
    """Synchronise and read the workspace's device error record (status code)."""
    return int(load_library().kla_workspace_check(
        _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)))


# ---- allocation helpers (torch memory only; the compute is the ABI call) ----

def alloc_workspace(B, T, H, dk, dv, chunk=64, io=KLA_IO_BF16, device="cuda",
                    segments=0) -> torch.Tensor:
    """Workspace for kla_chunk_fwd (segments=0) or kla_chunk_fwd_scan."""
    n = kla_chunk_fwd_scan_workspace_bytes(B, T, H, dk, dv, chunk, io, segments)
    if n == 0:
        raise KlaError(KLA_ERR_UNSUPPORTED, "kla_chunk_fwd_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def chunk_fwd(q, k, v, g, eta, eps=1e-6, h0=None, output_final_state=True, chunk=64,
              workspace=None, stream=None, beta=KLA_BETA_KACZMARZ):
    """Allocate o (and hT) and run kla_chunk_fwd (kla_chunk_fwd_ex when ``beta`` is
    KLA_BETA_DIRECT: eta is then the step size itself).  Returns (o, hT or None)."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device) if output_final_state else None
    if workspace is None:
        workspace = alloc_workspace(B, T, H, dk, dv, chunk, _io_of(q), q.device)
    if beta == KLA_BETA_KACZMARZ:
        kla_chunk_fwd(q, k, v, g, eta, eps, h0, o, hT, workspace, chunk, stream)
    else:
        kla_chunk_fwd_ex(q, k, v, g, eta, eps, h0, o, hT, workspace, beta=beta, chunk=chunk,
                         stream=stream)
    return o, hT


def chunk_bwd(q, k, v, g, eta, grad_o, grad_hT=None, eps=1e-6, h0=None, beta=KLA_BETA_KACZMARZ,
              workspace=None, stream=None):
    """Allocate the gradients and run kla_chunk_bwd.  Returns a dict with
    dq, dk, dv, dg, deta and dh0."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    out = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
               dg=torch.empty_like(g), deta=torch.empty_like(eta),
               dh0=torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device))
    if workspace is None:
        n = kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv, 64, _io_of(q))
        if n == 0:
            raise KlaError(KLA_ERR_UNSUPPORTED, "kla_chunk_bwd_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    kla_chunk_bwd(q, k, v, g, eta, eps, h0, grad_o, grad_hT, out["dq"], out["dk"], out["dv"],
                  out["dg"], out["deta"], out["dh0"], workspace, beta=beta, stream=stream)
    return out


class KLAChunk(torch.autograd.Function):
    """(o, hT) = KLA over a chunked sequence, differentiable in every input.

    Forward runs kla_chunk_fwd_ex, backward kla_chunk_bwd; no state is kept
    between them beyond the inputs."""

    @staticmethod
    def forward(ctx, q, k, v, g, eta, h0, eps, beta):
        B, T, H, dk = k.shape
        dv = v.shape[-1]
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
        hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
        ws = alloc_workspace(B, T, H, dk, dv, 64, _io_of(q), q.device)
        kla_chunk_fwd_ex(q, k, v, g, eta, eps, h0, o, hT, ws, beta=beta)
        ctx.save_for_backward(q, k, v, g, eta, h0)
        ctx.eps, ctx.beta = eps, beta
        return o, hT

    @staticmethod
    def backward(ctx, do, dhT):
        q, k, v, g, eta, h0 = ctx.saved_tensors
        do = torch.zeros_like(q[..., :1].expand(*q.shape[:3], v.shape[-1])) if do is None else do
        grads = chunk_bwd(q, k, v, g, eta, do.contiguous(),
                          None if dhT is None else dhT.contiguous(), ctx.eps, h0, ctx.beta)
        return (grads["dq"], grads["dk"], grads["dv"], grads["dg"], grads["deta"],
                grads["dh0"] if h0 is not None else None, None, None)


def kla_chunk(q, k, v, g, eta, eps=1e-6, h0=None, beta=KLA_BETA_KACZMARZ):
    """Differentiable chunkwise KLA: returns (o, hT) and supports .backward()."""
    return KLAChunk.apply(q.contiguous(), k.contiguous(), v.contiguous(), g.contiguous(),
                          eta.contiguous(), None if h0 is None else h0.contiguous(), float(eps),
                          int(beta))


def psd_features(x, d_out, stream=None):
    """Allocate and return the DeltaKATA features of x ([..., p] -> [..., d_out])."""
    y = torch.empty(x.shape[:-1] + (d_out,), dtype=x.dtype, device=x.device)
    kla_psd_features(x.contiguous(), y, stream)
    return y


class PSDFeatures(torch.autograd.Function):
    """psi(u) = u u^T as a vector (kla_psd_features), differentiable."""

    @staticmethod
    def forward(ctx, x, d_out):
        x = x.contiguous()
        ctx.save_for_backward(x)
        return psd_features(x, d_out)

    @staticmethod
    def backward(ctx, gy):
        (x,) = ctx.saved_tensors
        gx = torch.empty_like(x)
        kla_psd_features_bwd(x, gy.contiguous(), gx)
        return gx, None


class DeltaKATAFused(torch.autograd.Function):
    """DeltaKATA with 128 features through kla_deltakata_fwd: the forward forms
    the features inside the prefill; the backward forms them again
    (kla_psd_features), runs kla_chunk_bwd on them and maps the feature
    gradients back with kla_psd_features_bwd."""

    @staticmethod
    def forward(ctx, q, k, v, g, eta, h0, eps, beta):
        B, T, H, p = k.shape
        dv = v.shape[-1]
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
        hT = torch.empty((B, H, 128, dv), dtype=torch.float32, device=q.device)
        n = kla_deltakata_fwd_workspace_bytes(B, T, H, p, dv, 64, _io_of(q))
        if n == 0:
            raise KlaError(KLA_ERR_UNSUPPORTED, "kla_deltakata_fwd_workspace_bytes")
        ws = torch.empty(n, dtype=torch.uint8, device=q.device)
        kla_deltakata_fwd(q, k, v, g, eta, eps, h0, o, hT, ws, beta=beta)
        ctx.save_for_backward(q, k, v, g, eta, h0)
        ctx.eps, ctx.beta = eps, beta
        return o, hT

    @staticmethod
    def backward(ctx, do, dhT):
        q, k, v, g, eta, h0 = ctx.saved_tensors
        fq, fk = psd_features(q, 128), psd_features(k, 128)
        do = torch.zeros_like(v) if do is None else do
        grads = chunk_bwd(fq, fk, v, g, eta, do.contiguous(),
                          None if dhT is None else dhT.contiguous(), ctx.eps, h0, ctx.beta)
        gq, gk = torch.empty_like(q), torch.empty_like(k)
        kla_psd_features_bwd(q, grads["dq"], gq)
        kla_psd_features_bwd(k, grads["dk"], gk)
        return (gq, gk, grads["dv"], grads["dg"], grads["deta"],
                grads["dh0"] if h0 is not None else None, None, None)


def deltakata(q, k, v, g, eta, eps=1e-6, h0=None, d_feat=None, beta=KLA_BETA_KACZMARZ):
    """DeltaKATA: the KLA recurrence on the rank-one PSD features of q and k.

    q, k [B,T,H,p] with p(p+1)/2 <= d_feat in {64, 128} (default: the smaller
    that fits); v [B,T,H,dv].  Differentiable; returns (o, hT).  With 128
    features, bf16 and d_v = 128 the features are formed inside the prefill
    (DeltaKATAFused); otherwise kla_psd_features writes them first."""
    B, T, H, p = k.shape
    if d_feat is None:
        d_feat = 64 if p * (p + 1) // 2 <= 64 else 128
    if (d_feat == 128 and q.dtype == torch.bfloat16 and
            kla_deltakata_fwd_workspace_bytes(B, T, H, p, v.shape[-1], 64, KLA_IO_BF16) > 0):
        return DeltaKATAFused.apply(q.contiguous(), k.contiguous(), v.contiguous(), g.contiguous(),
                                    eta.contiguous(), None if h0 is None else h0.contiguous(),
                                    float(eps), int(beta))
    return kla_chunk(PSDFeatures.apply(q, d_feat), PSDFeatures.apply(k, d_feat), v, g, eta, eps,
                     h0, beta)


def loglinear_fwd(q, k, v, g, eta, lam, eps=1e-6, beta=KLA_BETA_KACZMARZ, workspace=None,
                  stream=None):
    """Allocate o and run kla_loglinear_fwd.  Returns o."""
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if workspace is None:
        n = kla_loglinear_workspace_bytes(B, T, H, dk, dv, 64, _io_of(q))
        if n == 0:
            raise KlaError(KLA_ERR_UNSUPPORTED, "kla_loglinear_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    kla_loglinear_fwd(q, k, v, g, eta, lam, eps, o, workspace, beta=beta, stream=stream)
    return o


def decode_step(q, k, v, g, eta, S, eps=1e-6, stream=None, beta=KLA_BETA_KACZMARZ):
    """Run kla_decode_step (with the step size chosen by ``beta``); S is updated in
    place.  Returns o."""
    o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    kla_decode_step(q, k, v, g, eta, eps, S, o, stream, beta=beta)
    return o


__all__ = [
    "kla_chunk_fwd_workspace_bytes", "kla_chunk_fwd", "kla_chunk_fwd_noalloc",
    "kla_chunk_fwd_noalloc_check", "kla_decode_step",
    "kla_chunk_fwd_scan", "kla_chunk_fwd_scan_workspace_bytes", "kla_chunk_fwd_auto_segments",
    "kla_chunk_fwd_ex", "kla_decode_step_ex", "KLA_BETA_KACZMARZ", "KLA_BETA_DIRECT",
    "kla_chunk_bwd", "kla_chunk_bwd_workspace_bytes", "chunk_bwd", "kla_chunk", "KLAChunk",
    "kla_psd_features", "kla_psd_features_bwd", "psd_features", "PSDFeatures", "deltakata",
    "kla_deltakata_fwd_workspace_bytes", "kla_deltakata_fwd", "DeltaKATAFused",
    "kla_loglinear_num_levels", "kla_loglinear_workspace_bytes", "kla_loglinear_fwd", "loglinear_fwd",
    "kla_loglinear_decode_step",
    "kla_workspace_check",
    "kla_status_string", "chunk_fwd", "decode_step", "alloc_workspace", "load_library",
    "KlaError", "EXPORTED_SYMBOLS", "KLA_IO_BF16", "KLA_IO_FP32",
]
