"""fp64 CPU restatement of the chunk algebra -- TEST INFRASTRUCTURE ONLY.

Only ``tests/`` imports this module.  It shares no code with the CUDA library
or with the sequential loop of ``kla_oracle.c``: it is a second, independent
derivation of the same results, in the chunked form the kernels compute, and
the tests hold it to the sequential oracle at 1e-12.  What it pins is the
algebra itself (the equations every kernel implements), independently of the
bf16/fp32 tolerances of the GPU parity tests.

Sources.  "KLA: Kaczmarz Linear Attention" (gist.science/ko/paper/2605.08587),
sections "KLA update rule" (beta_t = eta_t / (||k_t||^2 + eps), the delta
update) and "Implementation" (the GDN chunkwise solver is kept; only its
diagonal coefficient matrix becomes B = Diag(beta)).  The pages print no
chunk equations; the ones below come from unrolling the recurrence inside a
chunk of C tokens with local inclusive log-decay cumsum gam_r, Gam_r =
exp(gam_r), start state S0:

    D_rs = exp(gam_r - gam_s) (s <= r),  A = strict_lower(diag(beta) (D o K K^T))
    T = (I + A)^{-1},  U = T diag(beta) V,  Wk = T diag(beta Gam) K
    W = U - Wk S0
    O = diag(Gam) Q S0 + P W,            P = D o (Q K^T)   (s <= r)
    S1 = Gam_C S0 + K~^T W,              K~ = diag(exp(gam_C - gam_r)) K

The chunk-level scan ("Kernelized Linear Attention" page, section 2.3: the
inter-chunk state by an associative scan; "Higher-order Linear Attention"
page, section 4: a scan over segment summaries equals the serial recurrence)
uses that the chunk map is affine in S0: S1 = M S0 + N with
M = Gam_C I - K~^T Wk, N = K~^T U.

The Log-Linear form ("Log-Linear Attention", technical summary section 2)
keeps one state per Fenwick bucket and weighs each bucket's readout by
lambda_t^(level).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------- one chunk

def chunk_quantities(K, V, g, eta, eps, beta_direct=False):
    """State-independent quantities of one chunk (rows are its tokens).

    Returns a dict with gam, Gam, beta, D (inclusive decay mask), A, T, U, Wk
    and sc = exp(gam_C - gam_r)."""
    n = K.shape[0]
    gam = np.cumsum(g)
    Gam = np.exp(gam)
    kk = np.einsum("rd,rd->r", K, K)
    beta = eta.copy() if beta_direct else eta / (kk + eps)
    diff = gam[:, None] - gam[None, :]
    lower = np.tril(np.ones((n, n), dtype=bool))
    D = np.where(lower, np.exp(np.where(lower, diff, 0.0)), 0.0)
    A = np.tril(beta[:, None] * D * (K @ K.T), -1)
    T = np.linalg.inv(np.eye(n) + A)
    U = T @ (beta[:, None] * V)
    Wk = T @ ((beta * Gam)[:, None] * K)
    sc = np.exp(gam[-1] - gam)
    return dict(gam=gam, Gam=Gam, beta=beta, D=D, A=A, T=T, U=U, Wk=Wk, sc=sc)


def chunk_step(Q, K, V, g, eta, eps, S0, beta_direct=False, kernel_forms=False):
    """Outputs and end state of one chunk from its start state S0.

    ``kernel_forms`` evaluates the decay factors the way the tensor-core
    kernels do: when the chunk's decay span gam_0 - gam_last is at most 80,
    exp(gam_r - gam_s) = u_r w_s about the middle token m (u_r = exp(gam_r -
    gam_m), w_s = exp(gam_m - gam_s)), and P W = P' Wt with
    P'_rs = exp(gam_r - gam_C) (q_r . k_s) and Wt = diag(exp(gam_C - gam_s)) W
    (the output's in-chunk part riding in the state product); otherwise each
    factor is one exponential and P W is formed directly."""
    cq = chunk_quantities(K, V, g, eta, eps, beta_direct)
    n = K.shape[0]
    W = cq["U"] - cq["Wk"] @ S0
    QK = Q @ K.T
    if kernel_forms and (cq["gam"][0] - cq["gam"][-1]) <= 80.0:
        gam = cq["gam"]
        m = n // 2 - 1 if n > 1 else 0
        u = np.exp(gam - gam[m])
        w = np.exp(gam[m] - gam)
        lower = np.tril(np.ones((n, n), dtype=bool))
        Pp = np.where(lower, np.exp(gam - gam[-1])[:, None] * QK, 0.0)
        Wt = cq["sc"][:, None] * W
        PW = Pp @ Wt
        # the factorised mask reproduces D exactly in exact arithmetic
        Dfac = np.where(lower, u[:, None] * w[None, :], 0.0)
        A = np.tril(cq["beta"][:, None] * Dfac * (K @ K.T), -1)
        assert np.allclose(A, cq["A"], rtol=1e-12, atol=1e-300)
    else:
        PW = (cq["D"] * QK) @ W
    O = cq["Gam"][:, None] * (Q @ S0) + PW
    S1 = cq["Gam"][-1] * S0 + (cq["sc"][:, None] * K).T @ W
    return O, S1


def chunk_map(K, V, g, eta, eps, beta_direct=False):
    """The chunk's affine map S1 = M S0 + N (M: dk x dk, N: dk x dv)."""
    cq = chunk_quantities(K, V, g, eta, eps, beta_direct)
    Kt = cq["sc"][:, None] * K
    M = cq["Gam"][-1] * np.eye(K.shape[1]) - Kt.T @ cq["Wk"]
    N = Kt.T @ cq["U"]
    return M, N


# ------------------------------------------------------------ whole inputs

def _bounds(T, C):
    return [(t0, min(t0 + C, T)) for t0 in range(0, T, C)]


def chunk_forward(q, k, v, g, eta, eps, h0=None, *, C=64, beta_direct=False, kernel_forms=False):
    """Chunkwise forward over [B, T, H, d] inputs; the last chunk may be short.
    Returns (o [B,T,H,dv], hT [B,H,dk,dv])."""
    q, k, v, g, eta, h0 = map(_f64, (q, k, v, g, eta, h0))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].copy()
            for t0, t1 in _bounds(T, C):
                o[b, t0:t1, h], S = chunk_step(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h],
                                               g[b, t0:t1, h], eta[b, t0:t1, h], eps, S, beta_direct,
                                               kernel_forms)
            hT[b, h] = S
    return o, hT


def chunk_scan_forward(q, k, v, g, eta, eps, h0=None, *, C=64, runs=2, beta_direct=False):
    """The chunk-level scan: the chunks of each head split into ``runs``
    consecutive runs; each run's affine map [N | M] is the recurrence started
    from [0 | I] (values entering only the N half), the runs' start states
    follow from one sequential pass S_{j+1} = M_j S_j + N_j, and each run is
    then replayed from its start state for its outputs."""
    q, k, v, g, eta, h0 = map(_f64, (q, k, v, g, eta, h0))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    bounds = _bounds(T, C)
    per = -(-len(bounds) // runs) if bounds else 1
    groups = [bounds[i:i + per] for i in range(0, len(bounds), per)]
    o = np.zeros((B, T, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            maps = []
            for grp in groups:
                Nacc = np.zeros((dk, dv))
                Macc = np.eye(dk)
                for t0, t1 in grp:
                    M, N = chunk_map(k[b, t0:t1, h], v[b, t0:t1, h], g[b, t0:t1, h],
                                     eta[b, t0:t1, h], eps, beta_direct)
                    Nacc = M @ Nacc + N
                    Macc = M @ Macc
                maps.append((Macc, Nacc))
            starts = [np.zeros((dk, dv)) if h0 is None else h0[b, h].copy()]
            for Mj, Nj in maps:
                starts.append(Mj @ starts[-1] + Nj)
            for grp, S in zip(groups, starts):
                for t0, t1 in grp:
                    o[b, t0:t1, h], S = chunk_step(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h],
                                                   g[b, t0:t1, h], eta[b, t0:t1, h], eps, S, beta_direct)
            hT[b, h] = starts[-1]
    return o, hT


# ---------------------------------------------------------------- backward

def _chunk_backward(Q, K, V, g, eta, eps, S0, dO, dS1, beta_direct):
    """Reverse mode of chunk_step: returns dQ, dK, dV, dg, deta, dS0."""
    n = K.shape[0]
    gam = np.cumsum(g)
    Gam = np.exp(gam)
    kk = np.einsum("rd,rd->r", K, K)
    den = kk + eps
    beta = eta.copy() if beta_direct else eta / den
    lower = np.tril(np.ones((n, n), dtype=bool))
    strict = np.tril(np.ones((n, n), dtype=bool), -1)
    D = np.where(lower, np.exp(np.where(lower, gam[:, None] - gam[None, :], 0.0)), 0.0)
    G = K @ K.T
    A = np.where(strict, beta[:, None] * D * G, 0.0)
    T = np.linalg.inv(np.eye(n) + A)
    KS = K @ S0
    E = V - Gam[:, None] * KS                  # X = diag(beta) E
    X = beta[:, None] * E
    W = T @ X
    QK = Q @ K.T
    P = D * QK
    sc = np.exp(gam[-1] - gam)
    Kt = sc[:, None] * K

    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dGam = np.zeros(n)
    dD = np.zeros((n, n))
    dsc = np.zeros(n)
    dbeta = np.zeros(n)
    # S1 = Gam_C S0 + Kt^T W
    dS0 = Gam[-1] * dS1
    dGamC = np.sum(S0 * dS1)
    dW = Kt @ dS1
    dKt = W @ dS1.T
    dK += sc[:, None] * dKt
    dsc += np.einsum("rd,rd->r", K, dKt)
    # O = diag(Gam) Q S0 + P W
    QS = Q @ S0
    dGam += np.einsum("rj,rj->r", QS, dO)
    dQ += Gam[:, None] * (dO @ S0.T)
    dS0 += (Gam[:, None] * Q).T @ dO
    dP = np.where(lower, dO @ W.T, 0.0)
    dW += P.T @ dO
    dD += dP * QK
    dQK = dP * D
    dQ += dQK @ K
    dK += dQK.T @ Q
    # W = T X, (I + A) W = X
    dX = T.T @ dW
    dA = np.where(strict, -dX @ W.T, 0.0)
    # X = diag(beta) (V - diag(Gam) K S0)
    dbeta += np.einsum("rj,rj->r", dX, E)
    dE = beta[:, None] * dX
    dV = dE
    dGam += -np.einsum("rj,rj->r", KS, dE)
    dKS = -Gam[:, None] * dE
    dK += dKS @ S0.T
    dS0 += K.T @ dKS
    # A = strict(diag(beta) (D o G))
    dbeta += np.einsum("rs,rs->r", dA, D * G)
    dD += dA * beta[:, None] * G
    dG = dA * beta[:, None] * D
    dK += (dG + dG.T) @ K
    # decays: D_rs = exp(gam_r - gam_s), Gam_r = exp(gam_r), sc_r = exp(gam_C - gam_r)
    dgam = np.zeros(n)
    t = dD * D
    dgam += t.sum(axis=1) - t.sum(axis=0)
    dgam += dGam * Gam
    dgam[-1] += dGamC * Gam[-1]
    dgam[-1] += np.sum(dsc * sc)
    dgam -= dsc * sc
    dg = np.cumsum(dgam[::-1])[::-1]
    # step size
    if beta_direct:
        deta = dbeta
    else:
        deta = dbeta / den
        dK += (-2.0 * beta * dbeta / den)[:, None] * K
    return dQ, dK, dV, dg, deta, dS0


def chunk_backward(q, k, v, g, eta, eps, h0, dout, dhT=None, *, C=64, beta_direct=False):
    """Gradients of chunk_forward's (o, hT) given dL/do and dL/dhT: the forward
    states at every chunk start, then the chunks in reverse order, the state
    gradient passed back through the transposed chunk maps."""
    q, k, v, g, eta, h0, dout, dhT = map(_f64, (q, k, v, g, eta, h0, dout, dhT))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               dg=np.zeros_like(g), deta=np.zeros_like(eta), dh0=np.zeros((B, H, dk, dv)))
    bounds = _bounds(T, C)
    for b in range(B):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].copy()
            starts = []
            for t0, t1 in bounds:
                starts.append(S)
                _, S = chunk_step(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h], g[b, t0:t1, h],
                                  eta[b, t0:t1, h], eps, S, beta_direct)
            dS = np.zeros((dk, dv)) if dhT is None else dhT[b, h].copy()
            for (t0, t1), S0 in reversed(list(zip(bounds, starts))):
                dQ, dK, dV, dgc, detac, dS = _chunk_backward(
                    q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h], g[b, t0:t1, h],
                    eta[b, t0:t1, h], eps, S0, dout[b, t0:t1, h], dS, beta_direct)
                out["dq"][b, t0:t1, h] = dQ
                out["dk"][b, t0:t1, h] = dK
                out["dv"][b, t0:t1, h] = dV
                out["dg"][b, t0:t1, h] = dgc
                out["deta"][b, t0:t1, h] = detac
            out["dh0"][b, h] = dS
    return out


# ---------------------------------------------------------------- Log-Linear

def _level(t, s):
    return 0 if t == s else (t ^ s).bit_length()


def loglinear_chunk_forward(q, k, v, g, eta, lam, eps, *, C=64, beta_direct=False):
    """Log-Linear gated delta rule by chunks of C = 2^m tokens (or one chunk
    of the whole sequence).  Inside a chunk a write of token s reaches o_t
    through (P T diag(beta))_ts v_s, weighted by lambda_t^(level(t, s)), with
    level(t, s) <= m.  Earlier chunks live in one state per set bit j of the
    chunk index c (chunks c' with floor(log2(c xor c')) = j, level m + 1 + j),
    each read out through the chunk's state-to-output map
    diag(Gam) Q S - P Wk S.  Between chunks c and c + 1, with b the lowest set
    bit of c + 1, the levels below b merge into level b together with chunk
    c's write, and the levels above b only take the chunk's transition."""
    q, k, v, g, eta, lam = map(_f64, (q, k, v, g, eta, lam))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    if C < T:
        assert C & (C - 1) == 0, "chunks of a power-of-two length"
    m = (C - 1).bit_length()          # in-chunk levels 0..m
    o = np.zeros((B, T, H, dv))
    bounds = _bounds(T, C)
    for b in range(B):
        for h in range(H):
            states = {}                  # bit j -> state of the chunks at level m + 1 + j
            for c, (t0, t1) in enumerate(bounds):
                Q, K, V = q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h]
                cq = chunk_quantities(K, V, g[b, t0:t1, h], eta[b, t0:t1, h], eps, beta_direct)
                n = t1 - t0
                P = cq["D"] * (Q @ K.T)
                Lam = np.array([[lam[b, t0 + r, h, _level(t0 + r, t0 + s)] if s <= r else 0.0
                                 for s in range(n)] for r in range(n)])
                O = ((P @ cq["T"]) * cq["beta"][None, :] * Lam) @ V
                for j, S in states.items():
                    read = cq["Gam"][:, None] * (Q @ S) - P @ (cq["Wk"] @ S)
                    O += lam[b, t0:t1, h, m + 1 + j][:, None] * read
                o[b, t0:t1, h] = O
                if c + 1 == len(bounds):
                    break
                Kt = cq["sc"][:, None] * K
                low = ((c + 1) & -(c + 1)).bit_length() - 1
                Msum = sum((S for j, S in states.items() if j < low), np.zeros((dk, dv)))
                new = {j: cq["Gam"][-1] * S - Kt.T @ (cq["Wk"] @ S)
                       for j, S in states.items() if j > low}
                new[low] = cq["Gam"][-1] * Msum + Kt.T @ (cq["U"] - cq["Wk"] @ Msum)
                states = new
    return o


def loglinear_decode(q, k, v, g, eta, lam, eps, *, beta_direct=False):
    """Log-Linear decoding one token at a time with O(log T) bucket states:
    at token t every non-empty state takes the transition a_t (I - beta_t k_t
    k_t^T); with b the lowest set bit of t, levels 0..b (token t-1 and the
    buckets below b) merge into level b + 1, which is empty beforehand; the
    token's write beta_t k_t v_t^T takes level 0.  o_t = sum_l lambda_t^(l)
    S_t^(l)^T q_t."""
    q, k, v, g, eta, lam = map(_f64, (q, k, v, g, eta, lam))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            levels = {}
            for t in range(T):
                kt, qt = k[b, t, h], q[b, t, h]
                if t > 0:
                    low = (t & -t).bit_length() - 1
                    merged = sum((levels.pop(l) for l in range(low + 1) if l in levels),
                                 np.zeros((dk, dv)))
                    assert low + 1 not in levels
                    levels[low + 1] = merged
                a = np.exp(g[b, t, h])
                beta = eta[b, t, h] if beta_direct else eta[b, t, h] / (kt @ kt + eps)
                for l in levels:
                    S = levels[l]
                    levels[l] = a * (S - beta * np.outer(kt, kt @ S))
                levels[0] = beta * np.outer(kt, v[b, t, h])
                o[b, t, h] = sum(lam[b, t, h, l] * (levels[l].T @ qt) for l in levels)
    return o


__all__ = ["chunk_quantities", "chunk_step", "chunk_map", "chunk_forward", "chunk_scan_forward",
           "chunk_backward", "loglinear_chunk_forward", "loglinear_decode"]


def loglinear_level_passes(q, k, v, g, eta, lam, eps, *, C=64, beta_direct=False, pair=False):
    """Log-Linear gated delta rule as independent passes of the ordinary
    chunked recurrence, one per level above the chunk.

    A token s is in bucket level l of token t > s when t and s first differ
    at bit l - 1: s lies in the first half and t in the second half of the
    aligned block of 2^l tokens that holds both.  So level l's contribution to
    o_t is the ordinary recurrence restarted from zero at the block's start,
    with writes from the first half only, read out at t after t's own
    transition, weighted by lambda_t^(l).  With C = 2^m, levels l > m have
    blocks of whole chunks: per block, the first-half chunks run the chunk
    step with their values, the second-half chunks run it with zero values
    (S1 = M S0, O = (diag(Gam) Q - P Wk) S0) and their outputs count.  Levels
    0..m stay inside a chunk: O_in = ((P T diag(beta)) o Lam) V.

    With ``pair``, levels 0..m+1 are taken over aligned pairs of chunks as
    one chunk of 2C tokens, built from the two chunks' own quantities: with
    A_21[r][s] = beta_r exp(gam_r - gam_s) (k_r . k_s) the block of A that
    couples them (gam running over both), the inverse of the block lower
    triangular I + A gives T diag(beta) = [[Tb_1, 0], [-Tb_2 A~_21 Tb_1,
    Tb_2]] with Tb_i = T_i diag(beta_i) and A_21 = diag(beta_2) A~_21; the
    passes then start at level m + 2."""
    q, k, v, g, eta, lam = map(_f64, (q, k, v, g, eta, lam))
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    assert C & (C - 1) == 0
    m = (C - 1).bit_length()
    L = (max(T, 1) - 1).bit_length() + 1
    o = np.zeros((B, T, H, dv))
    bounds = _bounds(T, C)
    for b in range(B):
        for h in range(H):
            if pair:
                for p0 in range(0, len(bounds), 2):
                    t0 = bounds[p0][0]
                    t1 = bounds[min(p0 + 1, len(bounds) - 1)][1]
                    n = t1 - t0
                    Q, K, V = q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h]
                    n1 = bounds[p0][1] - t0
                    c1 = chunk_quantities(K[:n1], V[:n1], g[b, t0:t0 + n1, h], eta[b, t0:t0 + n1, h], eps,
                                          beta_direct)
                    Tb = np.zeros((n, n))
                    Tb[:n1, :n1] = c1["T"] * c1["beta"][None, :]
                    gam = np.cumsum(g[b, t0:t1, h])
                    if n > n1:
                        c2 = chunk_quantities(K[n1:], V[n1:], g[b, t0 + n1:t1, h], eta[b, t0 + n1:t1, h], eps,
                                              beta_direct)
                        Tb2 = c2["T"] * c2["beta"][None, :]
                        At = np.exp(gam[n1:, None] - gam[None, :n1]) * (K[n1:] @ K[:n1].T)
                        Tb[n1:, n1:] = Tb2
                        Tb[n1:, :n1] = -Tb2 @ At @ Tb[:n1, :n1]
                    lower = np.tril(np.ones((n, n), dtype=bool))
                    P = np.where(lower, np.exp(np.where(lower, gam[:, None] - gam[None, :], 0.0)), 0.0) * (Q @ K.T)
                    Lam = np.array([[lam[b, t0 + r, h, _level(t0 + r, t0 + s)] if s <= r else 0.0
                                     for s in range(n)] for r in range(n)])
                    o[b, t0:t1, h] += ((P @ Tb) * Lam) @ V
            # in-chunk levels 0..m
            for t0, t1 in (() if pair else bounds):
                K, V, Q = k[b, t0:t1, h], v[b, t0:t1, h], q[b, t0:t1, h]
                cq = chunk_quantities(K, V, g[b, t0:t1, h], eta[b, t0:t1, h], eps, beta_direct)
                n = t1 - t0
                P = cq["D"] * (Q @ K.T)
                Lam = np.array([[lam[b, t0 + r, h, _level(t0 + r, t0 + s)] if s <= r else 0.0
                                 for s in range(n)] for r in range(n)])
                o[b, t0:t1, h] += ((P @ cq["T"]) * cq["beta"][None, :] * Lam) @ V
            # one pass per level above the chunk: blocks of 2^(l - 1 - m) chunks per half
            for lev in range(m + 2 if pair else m + 1, L):
                half = 1 << (lev - 1 - m)
                for blk0 in range(0, len(bounds), 2 * half):
                    S = np.zeros((dk, dv))
                    for ci in range(blk0, min(blk0 + 2 * half, len(bounds))):
                        t0, t1 = bounds[ci]
                        writes = ci < blk0 + half
                        Vc = v[b, t0:t1, h] if writes else np.zeros_like(v[b, t0:t1, h])
                        O, S = chunk_step(q[b, t0:t1, h], k[b, t0:t1, h], Vc, g[b, t0:t1, h],
                                          eta[b, t0:t1, h], eps, S, beta_direct)
                        if not writes:
                            o[b, t0:t1, h] += lam[b, t0:t1, h, lev][:, None] * O
    return o
