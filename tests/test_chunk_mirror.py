"""The chunk algebra every kernel implements, pinned to the sequential oracle
in fp64.

``oracle/chunk_mirror.py`` restates the chunkwise form (the GDN chunk solver
with B = Diag(beta), "KLA: Kaczmarz Linear Attention", section
"Implementation"), the chunk-level scan of affine chunk maps ("Kernelized
Linear Attention" page, section 2.3; "Higher-order Linear Attention" page,
section 4), the reverse mode of the chunk algebra, and the Log-Linear
chunked carry and decoding ("Log-Linear Attention", technical summary
section 2).  Each is held to the sequential fp64 oracle at 1e-12 (relative to
the largest reference entry) over chunk lengths 1, 16, 64 and T, ragged
sequence lengths and a nonzero start state, so that a wrong term too small
to show at bf16 precision still fails here.
"""
import numpy as np
import pytest

import oracle
from oracle import chunk_mirror as cm
from tests.test_oracle_pins import _rand_inputs

TOL = 1e-12


def _rel(x, ref):
    ref = np.asarray(ref)
    return float(np.abs(np.asarray(x) - ref).max() / max(np.abs(ref).max(), 1e-300))


def _case(seed, B=2, T=150, H=2, dk=12, dv=9, knorm=(0.25, 4.0), h0_std=0.3, gates="random"):
    rng = np.random.default_rng(seed)
    return _rand_inputs(rng, B, T, H, dk, dv, knorm=knorm, h0_std=h0_std, gates=gates)


@pytest.mark.parametrize("C", [1, 16, 64, "T"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 150])
@pytest.mark.parametrize("direct", [False, True])
def test_chunk_forward_equals_the_sequential_loop(C, T, direct):
    q, k, v, g, eta, h0 = _case(100 + T, T=T, knorm=(0.5, 1.2) if direct else (0.25, 4.0))
    eps = 1e-6
    o_ref, h_ref = oracle.kla_oracle_forward(q, k, v, g, eta, eps, h0, beta_direct=direct)
    o, hT = cm.chunk_forward(q, k, v, g, eta, eps, h0, C=T if C == "T" else C, beta_direct=direct)
    assert _rel(o, o_ref) <= TOL
    assert _rel(hT, h_ref) <= TOL


@pytest.mark.parametrize("T", [64, 130, 200])
def test_kernel_decay_forms_equal_the_sequential_loop(T):
    """The factorised decay (u_r w_s about the middle token) and P W = P' Wt,
    used by the tensor-core kernels when a chunk's decay span is at most 80;
    strong decay (spans above 80) takes the direct branch in the same call."""
    q, k, v, g, eta, h0 = _case(7 + T, T=T, dk=16, dv=8)
    g = g.copy()
    g[:, 64:128] *= 12.0          # the second chunk's span far above 80
    o_ref, h_ref = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    o, hT = cm.chunk_forward(q, k, v, g, eta, 1e-6, h0, C=64, kernel_forms=True)
    assert _rel(o, o_ref) <= TOL
    assert _rel(hT, h_ref) <= TOL


def test_projection_workload_shape():
    """Unit decay and eta = 1, eps = 0 (the projection workload): the chunk
    form keeps S_t^T k_t = v_t at every chunk end."""
    q, k, v, g, eta, h0 = _case(5, B=1, T=128, H=1, dk=32, dv=8, knorm=(0.1, 10.0),
                                gates="projection", h0_std=0.01)
    o_ref, h_ref = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0)
    o, hT = cm.chunk_forward(q, k, v, g, eta, 0.0, h0, C=64)
    assert _rel(o, o_ref) <= 1e-11
    assert _rel(hT, h_ref) <= 1e-11
    assert np.allclose(hT[0, 0].T @ k[0, -1, 0], v[0, -1, 0], atol=1e-9)


def test_orthogonal_keys_give_the_identity_solve():
    """Mutually orthogonal keys inside a chunk: K K^T is diagonal, so A = 0 and
    T = (I + A)^{-1} = I; U = diag(beta) V and Wk = diag(beta Gam) K."""
    rng = np.random.default_rng(3)
    n, d = 16, 32
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    K = Qm[:n] * rng.uniform(0.5, 2.0, (n, 1))
    V = rng.standard_normal((n, 7))
    g = -rng.uniform(0.0, 0.3, n)
    eta = rng.uniform(0.2, 1.0, n)
    cq = cm.chunk_quantities(K, V, g, eta, 1e-6)
    assert np.abs(cq["A"]).max() < 1e-13
    assert np.allclose(cq["T"], np.eye(n), atol=1e-13)
    assert np.allclose(cq["U"], cq["beta"][:, None] * V, atol=1e-13)
    assert np.allclose(cq["Wk"], (cq["beta"] * cq["Gam"])[:, None] * K, atol=1e-13)


def test_chunk_map_is_the_affine_transition():
    """S1 = M S0 + N for any start state: the map of one chunk applied to two
    start states differs by M times their difference."""
    q, k, v, g, eta, _ = _case(9, B=1, T=64, H=1, dk=10, dv=6)
    Q, K, V, gg, ee = q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], eta[0, :, 0]
    M, N = cm.chunk_map(K, V, gg, ee, 1e-6)
    rng = np.random.default_rng(1)
    for _ in range(3):
        S0 = rng.standard_normal((10, 6))
        _, S1 = cm.chunk_step(Q, K, V, gg, ee, 1e-6, S0)
        assert _rel(S1, M @ S0 + N) <= TOL


@pytest.mark.parametrize("runs", [1, 2, 3, 5, 64])
@pytest.mark.parametrize("C", [16, 64])
def test_chunk_scan_equals_the_sequential_loop(runs, C):
    q, k, v, g, eta, h0 = _case(40 + runs, T=333, dk=8, dv=6)
    o_ref, h_ref = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    o, hT = cm.chunk_scan_forward(q, k, v, g, eta, 1e-6, h0, C=C, runs=runs)
    assert _rel(o, o_ref) <= 1e-11
    assert _rel(hT, h_ref) <= 1e-11


@pytest.mark.parametrize("C", [1, 16, 64, "T"])
@pytest.mark.parametrize("T", [1, 65, 130])
@pytest.mark.parametrize("direct", [False, True])
def test_chunk_backward_equals_the_sequential_reverse_mode(C, T, direct):
    q, k, v, g, eta, h0 = _case(200 + T, B=1, T=T, dk=8, dv=5,
                                knorm=(0.5, 1.2) if direct else (0.25, 4.0))
    rng = np.random.default_rng(T)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal((1, 2, 8, 5))
    eps = 1e-3
    ref = oracle.kla_oracle_backward(q, k, v, g, eta, eps, h0, dout, dhT, beta_direct=direct)
    got = cm.chunk_backward(q, k, v, g, eta, eps, h0, dout, dhT, C=T if C == "T" else C,
                            beta_direct=direct)
    for name in ("dq", "dk", "dv", "dg", "deta", "dh0"):
        assert _rel(got[name], ref[name]) <= 1e-10, name


def test_chunk_backward_without_start_state_and_state_gradient():
    q, k, v, g, eta, _ = _case(77, B=1, T=100, dk=6, dv=4, h0_std=0.0)
    dout = np.random.default_rng(2).standard_normal(v.shape)
    ref = oracle.kla_oracle_backward(q, k, v, g, eta, 1e-6, None, dout, None)
    got = cm.chunk_backward(q, k, v, g, eta, 1e-6, None, dout, None, C=64)
    for name in ("dq", "dk", "dv", "dg", "deta", "dh0"):
        assert _rel(got[name], ref[name]) <= 1e-10, name


@pytest.mark.parametrize("C", [1, 4, 16, 64, "T"])
@pytest.mark.parametrize("T", [1, 37, 64, 200])
@pytest.mark.parametrize("direct", [False, True])
def test_loglinear_chunked_carry_equals_the_by_origin_oracle(C, T, direct):
    q, k, v, g, eta, _ = _case(300 + T, B=1, T=T, dk=6, dv=4,
                               knorm=(0.5, 1.2) if direct else (0.25, 4.0), h0_std=0.0)
    L = oracle.loglinear_num_levels(T) + 1
    lam = np.random.default_rng(T + 1).uniform(0.2, 1.5, (1, T, 2, L))
    ref = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 1e-6, beta_direct=direct)
    got = cm.loglinear_chunk_forward(q, k, v, g, eta, lam, 1e-6, C=T if C == "T" else C,
                                     beta_direct=direct)
    assert _rel(got, ref) <= 1e-11


@pytest.mark.parametrize("direct", [False, True])
def test_loglinear_decoding_equals_the_by_origin_oracle(direct):
    T = 150
    q, k, v, g, eta, _ = _case(500, B=1, T=T, dk=6, dv=4,
                               knorm=(0.5, 1.2) if direct else (0.25, 4.0), h0_std=0.0)
    L = oracle.loglinear_num_levels(T)
    lam = np.random.default_rng(9).uniform(0.2, 1.5, (1, T, 2, L))
    ref = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 1e-6, beta_direct=direct)
    got = cm.loglinear_decode(q, k, v, g, eta, lam, 1e-6, beta_direct=direct)
    assert _rel(got, ref) <= 1e-11


@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("T", [64, 130, 256, 333])
@pytest.mark.parametrize("direct", [False, True])
def test_loglinear_level_passes_equal_the_by_origin_oracle(C, T, direct):
    """The Log-Linear output as one ordinary chunked pass per level above the
    chunk (each aligned block restarted from zero, writes from its first half,
    outputs in its second half) plus the in-chunk levels."""
    q, k, v, g, eta, _ = _case(600 + T, B=1, T=T, dk=6, dv=4,
                               knorm=(0.5, 1.2) if direct else (0.25, 4.0), h0_std=0.0)
    L = oracle.loglinear_num_levels(T) + 1
    lam = np.random.default_rng(T + 7).uniform(0.2, 1.5, (1, T, 2, L))
    ref = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 1e-6, beta_direct=direct)
    got = cm.loglinear_level_passes(q, k, v, g, eta, lam, 1e-6, C=C, beta_direct=direct)
    assert _rel(got, ref) <= 1e-11


@pytest.mark.parametrize("C", [4, 16, 64])
@pytest.mark.parametrize("T", [64, 100, 130, 256, 333])
@pytest.mark.parametrize("direct", [False, True])
def test_loglinear_chunk_pairs_equal_the_by_origin_oracle(C, T, direct):
    """Levels 0..m+1 over aligned pairs of chunks, with the pair's
    T diag(beta) assembled from the two chunks' own (the block inverse), and
    the passes from level m + 2; ragged T leaves a pair with one chunk or a
    short second chunk."""
    q, k, v, g, eta, _ = _case(800 + T, B=1, T=T, dk=6, dv=4,
                               knorm=(0.5, 1.2) if direct else (0.25, 4.0), h0_std=0.0)
    L = oracle.loglinear_num_levels(T) + 1
    lam = np.random.default_rng(T + 9).uniform(0.2, 1.5, (1, T, 2, L))
    ref = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 1e-6, beta_direct=direct)
    got = cm.loglinear_level_passes(q, k, v, g, eta, lam, 1e-6, C=C, beta_direct=direct, pair=True)
    assert _rel(got, ref) <= 1e-11


# ------------------------------------------------------------------
# The tensor-core backward's arrangement of the chunk algebra (bf16 I/O,
# d_k = d_v = 128 in the library), restated in fp64: the carries form U from
# T diag(beta) and L = dO^T diag(Gam) Q themselves and keep W, dW, S0 and dS1;
# the gradient kernel stacks its products ([P' ; G], [X1 ; Y1], [dP ; -dA],
# [X2 ; Z5]) and takes dgamma's column sums separately.  Every step is an
# exact rewrite of the chunk reverse mode, so it must equal the oracle's
# sequential reverse mode to rounding.

def _tc_backward(q, k, v, g, eta, eps, h0, dout, dhT, C=64, beta_direct=False):
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), deta=np.zeros_like(eta), dh0=np.zeros((B, H, dk, dv)))
    for b in range(B):
        for h in range(H):
            recs, S = [], (np.zeros((dk, dv)) if h0 is None else h0[b, h].copy())
            for t0 in range(0, T, C):
                t1 = min(t0 + C, T)
                Q, K, V, O = q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h], dout[b, t0:t1, h]
                gam = np.cumsum(g[b, t0:t1, h])
                G = K @ K.T
                kk = np.diag(G).copy()
                beta = eta[b, t0:t1, h] if beta_direct else eta[b, t0:t1, h] / (kk + eps)
                Dm = np.exp(gam[:, None] - gam[None, :])
                n = len(gam)
                strict, incl = np.tril(np.ones((n, n)), -1), np.tril(np.ones((n, n)))
                At = strict * Dm * G                       # D o G, s < r
                Tm = np.linalg.inv(np.eye(n) + beta[:, None] * At)
                Wk = Tm @ ((beta * np.exp(gam))[:, None] * K)
                sc = np.exp(gam[-1] - gam)
                PT = np.triu(np.exp(gam[None, :] - gam[:, None]) * (K @ Q.T))   # P^T from K Q^T, s >= r
                # forward carry: D = -V^T Tb^T + S0^T Wk^T = -W^T
                W = -(-(V.T @ (Tm * beta[None, :]).T) + S.T @ Wk.T).T
                recs.append(dict(Q=Q, K=K, V=V, O=O, gam=gam, G=G, kk=kk, beta=beta, Dm=Dm, At=At, Tm=Tm,
                                 Wk=Wk, sc=sc, PT=PT, S0=S.copy(), W=W, n=n, strict=strict, incl=incl, t0=t0))
                S = np.exp(gam[-1]) * S + K.T @ (sc[:, None] * W)
            dS = np.zeros((dk, dv)) if dhT is None else dhT[b, h].copy()
            for r in reversed(recs):
                Q, K, V, O, gam, beta, Dm, n = r["Q"], r["K"], r["V"], r["O"], r["gam"], r["beta"], r["Dm"], r["n"]
                S0, W, Tm, At, Wk, sc = r["S0"], r["W"], r["Tm"], r["At"], r["Wk"], r["sc"]
                Gam = np.exp(gam)
                # reverse carry: D = dS1^T K^T, dW = diag(sc) D^T + P^T dO;  S_acc = dO^T diag(Gam) Q - dW^T Wk
                dW = sc[:, None] * (dS.T @ K.T).T + r["PT"] @ O
                dS1 = dS
                dS = np.exp(gam[-1]) * dS + (O.T @ (Gam[:, None] * Q) - dW.T @ Wk).T
                # gradient kernel, phase 1
                dX = Tm.T @ dW
                PG = np.vstack([Q, K]) @ K.T
                P = r["incl"] * Dm * PG[:n]
                At_ = r["strict"] * Dm * PG[n:]
                E1 = K @ S0
                Z1 = W @ dS1.T
                # phases 3 and 4
                XY = np.vstack([O, dX]) @ S0.T
                dPA = np.vstack([O, dX]) @ W.T
                E2 = At_ @ W
                e = V - Gam[:, None] * E1 - E2
                dbeta = (dX * e).sum(1)
                dgam = Gam * (Q * XY[:n]).sum(1) - Gam * beta * (K * XY[n:]).sum(1)
                z = sc * (K * Z1).sum(1)
                dgam -= z
                total = z.sum() + np.exp(gam[-1]) * (dS1 * S0).sum()
                dPm = r["incl"] * dPA[:n]
                dA = -r["strict"] * dPA[n:]
                dgam += (dPm * P).sum(1) - (dPm * P).sum(0)
                dgam += beta * (dA * At_).sum(1) - (beta[:, None] * dA * At_).sum(0)
                dPD = dPm * Dm
                F = beta[:, None] * r["strict"] * Dm * dA
                # phase 5: [X2 ; Z5] = [dPD ; F] K + [0 ; dPD^T] Q + [0 ; F^T] K
                Z = np.zeros((n, n))
                X2Z5 = np.vstack([dPD, F]) @ K + np.vstack([Z, dPD.T]) @ Q + np.vstack([Z, F.T]) @ K
                den = r["kk"] + eps
                vrs = np.zeros(n) if beta_direct else -2 * beta * dbeta / den
                dQ = Gam[:, None] * XY[:n] + X2Z5[:n]
                dK = -(Gam * beta)[:, None] * XY[n:] + sc[:, None] * Z1 + X2Z5[n:] + vrs[:, None] * K
                dgam[-1] += total
                t0, t1 = r["t0"], r["t0"] + n
                out["dq"][b, t0:t1, h] = dQ
                out["dk"][b, t0:t1, h] = dK
                out["dv"][b, t0:t1, h] = beta[:, None] * dX
                out["dg"][b, t0:t1, h] = np.cumsum(dgam[::-1])[::-1]
                out["deta"][b, t0:t1, h] = dbeta if beta_direct else dbeta / den
            out["dh0"][b, h] = dS
    return out


@pytest.mark.parametrize("C", [16, 64, "T"])
@pytest.mark.parametrize("T", [1, 65, 130])
@pytest.mark.parametrize("direct", [False, True])
def test_tensor_core_backward_arrangement_equals_the_sequential_reverse_mode(C, T, direct):
    q, k, v, g, eta, h0 = _case(300 + T, B=1, T=T, dk=8, dv=5,
                                knorm=(0.5, 1.2) if direct else (0.25, 4.0))
    rng = np.random.default_rng(3 + T)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal((1, 2, 8, 5))
    eps = 1e-3
    ref = oracle.kla_oracle_backward(q, k, v, g, eta, eps, h0, dout, dhT, beta_direct=direct)
    got = _tc_backward(*(np.asarray(x, np.float64) for x in (q, k, v, g, eta)), eps,
                       np.asarray(h0, np.float64), dout, dhT, C=T if C == "T" else C, beta_direct=direct)
    for name in ("dq", "dk", "dv", "dg", "deta", "dh0"):
        assert _rel(got[name], ref[name]) <= 1e-10, name
