"""fp64 CPU oracle for the KLA recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.

``kla_oracle_forward`` wraps the plain sequential C loop in ``kla_oracle.c``
(fp64, program order, no fast-math).  It follows "KLA: Kaczmarz Linear
Attention" (gist.science/ko/paper/2605.08587), section "KLA update rule":
beta_t = eta_t / (||k_t||^2 + eps), S_t = S~_{t-1} + beta_t k_t e_t^T with
e_t = v_t - S~_{t-1}^T k_t, S~_{t-1} = exp(g_t) S_{t-1}, and o_t = S_t^T q_t.
The decode-step oracle is the same loop with T = 1 and h0 = S.

Pins (all in ``tests/test_oracle_*.py``): the projection constraint
S_t^T k_t = v_t at eta=1, eps=0 (section "Theoretical derivation"); the
minimum-Frobenius-norm property against a least-squares solve; the exact
line search and the normalised-SGD step (section "Key properties"); the
beta=0 closed form; the no-erase mode against brute-force masked attention;
and a hand-worked two-token fixture under ``tests/golden/``.

``kla_oracle_backward`` is the reverse-mode derivative of the same loop
(every state kept, the step undone operation by operation), pinned by central
finite differences of ``kla_oracle_forward`` and by torch autograd.

``kla_oracle_psd_features`` is the rank-one PSD feature map of the KATA page
(psi(u) = u u^T as a vector), under which the same recurrence is DeltaKATA;
it is pinned by its inner-product identity and by numpy's outer product.

``kla_oracle_loglinear_forward`` is the Log-Linear gated delta rule (one
state per Fenwick bucket, weighted readout), written out by origin token.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kla_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkla_oracle.so")

NO_ERASE = 1
BETA_DIRECT = 2

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain IEEE fp64, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            f = lib.kla_oracle_forward
            dp = ctypes.POINTER(ctypes.c_double)
            i64 = ctypes.c_int64
            f.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp, dp,
                          i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int]
            f.restype = ctypes.c_int
            fb = lib.kla_oracle_backward
            fb.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp,
                           dp, dp, dp, dp, dp, dp,
                           i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int]
            fb.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy on the host
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def kla_oracle_forward(q, k, v, g, eta, eps, h0=None, *, no_erase=False,
                       return_states=False, threads=0, beta_direct=False):
    """Sequential fp64 forward over t for every (b, h).

    ``beta_direct``: beta_t = eta_t as given (the learned-scalar step size of
    Gated DeltaNet that the KLA page's sections "Problem statement" and
    "Methodology" contrast with the Kaczmarz step); eps is then unused.

    Shapes: q,k [B,T,H,dk]; v [B,T,H,dv]; g,eta [B,T,H]; h0 [B,H,dk,dv] or None.
    Returns (o [B,T,H,dv], hT [B,H,dk,dv]) and, with ``return_states``, also
    states [B,H,T,dk,dv] with states[b,h,t] = S_t (small inputs only).
    """
    q, k, v, g, eta, h0 = map(_f64, (q, k, v, g, eta, h0))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert q.shape == (B, T, H, dk) and v.shape == (B, T, H, dv)
    assert g.shape == (B, T, H) and eta.shape == (B, T, H)
    if h0 is not None:
        assert h0.shape == (B, H, dk, dv)
    o = np.zeros((B, T, H, dv), np.float64)
    hT = np.zeros((B, H, dk, dv), np.float64)
    states = np.zeros((B, H, T, dk, dv), np.float64) if return_states else None
    rc = _load().kla_oracle_forward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(eta), float(eps), _ptr(h0),
        _ptr(o), _ptr(hT), _ptr(states), B, T, H, dk, dv,
        (NO_ERASE if no_erase else 0) | (BETA_DIRECT if beta_direct else 0), int(threads))
    if rc != 0:
        raise RuntimeError(f"kla_oracle_forward failed with code {rc}")
    if return_states:
        return o, hT, states
    return o, hT


def kla_oracle_decode_step(q, k, v, g, eta, eps, S, *, beta_direct=False):
    """One recurrent decode step: the forward loop with T = 1, h0 = S.

    Shapes: q,k [B,H,dk]; v [B,H,dv]; g,eta [B,H]; S [B,H,dk,dv].
    Returns (o [B,H,dv], S_new [B,H,dk,dv]).
    """
    q, k, v, g, eta, S = map(_f64, (q, k, v, g, eta, S))
    o, hT = kla_oracle_forward(q[:, None], k[:, None], v[:, None], g[:, None],
                               eta[:, None], eps, S, beta_direct=beta_direct)
    return o[:, 0], hT


def kla_oracle_backward(q, k, v, g, eta, eps, h0, dout, dhT=None, *, beta_direct=False,
                        threads=0):
    """Gradients of ``kla_oracle_forward`` (fp64, sequential reverse mode).

    ``dout`` is dL/do [B,T,H,dv]; ``dhT`` is dL/dh_T [B,H,dk,dv] or None (zero).
    Returns a dict with dq, dk [B,T,H,dk], dv [B,T,H,dv], dg, deta [B,T,H] and
    dh0 [B,H,dk,dv] (the gradient of the start state, zero-state included).
    """
    q, k, v, g, eta, h0, dout, dhT = map(_f64, (q, k, v, g, eta, h0, dout, dhT))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert q.shape == (B, T, H, dk) and v.shape == (B, T, H, dv) and dout.shape == v.shape
    assert g.shape == (B, T, H) and eta.shape == (B, T, H)
    for s_ in (h0, dhT):
        assert s_ is None or s_.shape == (B, H, dk, dv)
    out = dict(dq=np.zeros((B, T, H, dk)), dk=np.zeros((B, T, H, dk)), dv=np.zeros((B, T, H, dv)),
               dg=np.zeros((B, T, H)), deta=np.zeros((B, T, H)), dh0=np.zeros((B, H, dk, dv)))
    rc = _load().kla_oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(eta), float(eps), _ptr(h0), _ptr(dout), _ptr(dhT),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["deta"]),
        _ptr(out["dh0"]), B, T, H, dk, dv, BETA_DIRECT if beta_direct else 0, int(threads))
    if rc != 0:
        raise RuntimeError(f"kla_oracle_backward failed with code {rc}")
    return out


def psd_feature_index(p: int):
    """The (i, j), i <= j, of each feature, row-major over the upper triangle."""
    return [(i, j) for i in range(p) for j in range(i, p)]


def kla_oracle_psd_features(x, d_out):
    """Rank-one PSD feature of each row u of x (shape [..., p]), as a vector.

    "Kernelized Linear Attention: breaking the capacity wall via symmetric
    cones", section 2.2: psi(u) = u u^T.  The symmetric matrix is written out
    as its upper triangle, row-major, with the off-diagonal entries scaled by
    sqrt(2) (so that the Frobenius inner product of two features is the dot
    product of their vectors), then padded with zeros to d_out >= p(p+1)/2.
    """
    x = _f64(x)
    p = x.shape[-1]
    idx = psd_feature_index(p)
    assert d_out >= len(idx)
    y = np.zeros(x.shape[:-1] + (d_out,), np.float64)
    for n, (i, j) in enumerate(idx):
        y[..., n] = x[..., i] * x[..., j] * (1.0 if i == j else np.sqrt(2.0))
    return y


def kla_oracle_psd_features_bwd(x, dy):
    """dL/dx given dL/dy for y = kla_oracle_psd_features(x, d_out): for the
    entry y = c x_i x_j, dx_i += c x_j dy and dx_j += c x_i dy (2 x_i dy on the
    diagonal)."""
    x, dy = _f64(x), _f64(dy)
    p = x.shape[-1]
    dx = np.zeros_like(x)
    for n, (i, j) in enumerate(psd_feature_index(p)):
        if i == j:
            dx[..., i] += 2.0 * x[..., i] * dy[..., n]
        else:
            c = np.sqrt(2.0)
            dx[..., i] += c * x[..., j] * dy[..., n]
            dx[..., j] += c * x[..., i] * dy[..., n]
    return dx


def loglinear_level(t: int, s: int) -> int:
    """Fenwick level of token s in the prefix of token t (s <= t): 0 for s = t,
    else one more than the highest bit in which t and s differ ("Log-Linear
    Attention", technical summary section 2: the prefix is split into buckets
    of exponentially growing size, recent tokens in the small ones)."""
    assert 0 <= s <= t
    return 0 if s == t else (t ^ s).bit_length()


def loglinear_num_levels(T: int) -> int:
    """Levels a sequence of T tokens uses: 1 + ceil(log2 T) (1 for T <= 1)."""
    return 1 + (max(T, 1) - 1).bit_length()


def kla_oracle_loglinear_forward(q, k, v, g, eta, lam, eps, *, beta_direct=False, no_erase=False):
    """Log-Linear gated delta rule, written out by origin token.

    "Log-Linear Attention", technical summary section 2: one state per Fenwick
    bucket and o_t = sum_l lambda_t^(l) q_t^T S_t^(l).  Read with the delta
    rule's transition A_t = a_t (I - beta_t k_t k_t^T) acting on every bucket
    and each write beta_s k_s v_s^T kept in the bucket of its token s:

        S_t^(l) = sum_{s <= t, level(t, s) = l} A_t ... A_{s+1} beta_s k_s v_s^T

    so that the buckets sum to the ordinary state.  A write's propagation only
    changes its key: x_s <- a_t (x_s - beta_t k_t (k_t . x_s)), and
    o_t = sum_s lambda_t^(level(t, s)) (q_t . x_s) v_s.  With ``no_erase`` the
    transition is a_t I and beta = 1 (linear attention: o = (Q K^T o M_H) V).
    Starts from a zero state.  lam: [B, T, H, L] with L >= loglinear_num_levels(T).
    """
    q, k, v, g, eta, lam = map(_f64, (q, k, v, g, eta, lam))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert lam.shape[:3] == (B, T, H) and lam.shape[3] >= loglinear_num_levels(T)
    o = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            X = np.zeros((T, dk))              # propagated keys of tokens 0..t
            for t in range(T):
                kt = k[b, t, h]
                a = np.exp(g[b, t, h])
                if no_erase:
                    beta = 1.0
                    X[:t] *= a
                else:
                    beta = eta[b, t, h] if beta_direct else eta[b, t, h] / (kt @ kt + eps)
                    X[:t] = a * (X[:t] - beta * np.outer(X[:t] @ kt, kt))
                X[t] = beta * kt
                # level(t, s) for s = 0..t: the bit length of t xor s (frexp's exponent)
                lev = np.frexp((t ^ np.arange(t + 1)).astype(np.float64))[1]
                w = lam[b, t, h][lev] * (X[:t + 1] @ q[b, t, h])
                o[b, t, h] = w @ v[b, :t + 1, h]
    return o


__all__ = ["build", "kla_oracle_forward", "kla_oracle_decode_step", "kla_oracle_backward",
           "kla_oracle_psd_features", "kla_oracle_psd_features_bwd", "psd_feature_index",
           "kla_oracle_loglinear_forward", "loglinear_level", "loglinear_num_levels",
           "NO_ERASE", "BETA_DIRECT"]
