"""Pins of the fp64 oracle against what the KLA page and the mathematics fix.

Page: "KLA: Kaczmarz Linear Attention" (gist.science/ko/paper/2605.08587).
  - section "Theoretical derivation": the write solves
    min 1/2 ||S - S~||_F^2 subject to S^T k = v; its solution is the
    orthogonal projection, step 1/||k||^2;
  - section "KLA update rule": beta = eta/(||k||^2 + eps), S = S~ + beta k e^T;
  - section "Key properties": at eta=1, eps=0 the step is the minimum-norm
    change, the exact line-search minimiser along the update direction and a
    normalised SGD step on the per-token loss.
Every test here checks the oracle against something other than itself: a
least-squares solve, a numerical line search, autograd, a closed form, a
brute-force O(T^2) masked attention, or a hand-worked fixture.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_inputs(rng, B, T, H, dk, dv, *, gates="random", knorm=(0.25, 4.0), h0_std=0.0):
    q = rng.standard_normal((B, T, H, dk))
    u = rng.standard_normal((B, T, H, dk))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    r = np.exp(rng.uniform(math.log(knorm[0]), math.log(knorm[1]), (B, T, H, 1)))
    k = u * r
    v = rng.standard_normal((B, T, H, dv))
    if gates == "projection":
        g = np.zeros((B, T, H))
        eta = np.ones((B, T, H))
    elif gates == "decay_only":
        g = -np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + 2.0)))
        eta = np.ones((B, T, H))
    else:
        g = -np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + 2.0)))
        eta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = rng.standard_normal((B, H, dk, dv)) * h0_std if h0_std > 0 else None
    return q, k, v, g, eta, h0


def _prev_states(states, h0, B, H, dk, dv):
    """S_{t-1} for every t (S_{-1} = h0 or 0)."""
    prev = np.empty_like(states)
    prev[:, :, 1:] = states[:, :, :-1]
    prev[:, :, 0] = h0 if h0 is not None else 0.0
    return prev


def test_golden_hand_two_tokens():
    vals = {}
    with open(os.path.join(GOLDEN, "hand_two_tokens.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    B, T, H, dk, dv = 1, 2, 1, 2, 3
    o, hT = oracle.kla_oracle_forward(
        vals["q"].reshape(B, T, H, dk), vals["k"].reshape(B, T, H, dk),
        vals["v"].reshape(B, T, H, dv), vals["g"].reshape(B, T, H),
        vals["eta"].reshape(B, T, H), float(vals["eps"][0]),
        vals["h0"].reshape(B, H, dk, dv))
    np.testing.assert_allclose(o.ravel(), vals["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(hT.ravel(), vals["hT"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("gates", ["projection", "decay_only"])
def test_projection_constraint_each_step(gates):
    """eta=1, eps=0: every step satisfies S_t^T k_t = v_t (to 1e-10)."""
    rng = np.random.default_rng(11)
    B, T, H, dk, dv = 2, 40, 2, 12, 7
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, gates=gates,
                                       knorm=(0.1, 10.0), h0_std=0.3)
    o, hT, st = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, return_states=True)
    kk = np.transpose(k, (0, 2, 1, 3))  # [B,H,T,dk]
    vv = np.transpose(v, (0, 2, 1, 3))
    lhs = np.einsum("bhtij,bhti->bhtj", st, kk)
    rel = np.abs(lhs - vv).max() / np.abs(vv).max()
    assert rel < 1e-10, rel
    np.testing.assert_array_equal(hT, st[:, :, -1])


def test_min_norm_change_matches_least_squares():
    """The update is the minimum-Frobenius-norm change satisfying the
    constraint: compare with numpy's min-norm least-squares solution of the
    linear system (I_dv kron k^T) vec(dS) = v - S~^T k, and check that dS is
    orthogonal to every D with D^T k = 0."""
    rng = np.random.default_rng(12)
    B, T, H, dk, dv = 1, 12, 1, 6, 4
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, gates="decay_only",
                                       knorm=(0.1, 10.0), h0_std=0.5)
    o, hT, st = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, return_states=True)
    prev = _prev_states(st, h0, B, H, dk, dv)
    for t in range(T):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = np.exp(g[0, t, 0]) * prev[0, 0, t]
        dS = st[0, 0, t] - St
        M = np.zeros((dv, dk * dv))
        for j in range(dv):
            for i in range(dk):
                M[j, i * dv + j] = kt[i]
        r = vt - St.T @ kt
        sol, *_ = np.linalg.lstsq(M, r, rcond=None)
        np.testing.assert_allclose(dS.ravel(), sol, rtol=1e-9, atol=1e-11)
        # orthogonality against the constraint's null space
        for _ in range(3):
            D = rng.standard_normal((dk, dv))
            D -= np.outer(kt, kt @ D) / (kt @ kt)
            assert abs(np.sum(dS * D)) < 1e-9 * np.linalg.norm(dS) * np.linalg.norm(D) + 1e-14


def test_exact_line_search():
    """eta=1, eps=0: the step length along k e^T minimises the per-token loss
    L(alpha) = 1/2 ||(S~ + alpha k e^T)^T k - v||^2 (found numerically)."""
    from scipy.optimize import minimize_scalar
    rng = np.random.default_rng(13)
    B, T, H, dk, dv = 1, 10, 1, 9, 5
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, gates="decay_only",
                                       knorm=(0.1, 10.0), h0_std=0.5)
    o, hT, st = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, return_states=True)
    prev = _prev_states(st, h0, B, H, dk, dv)
    for t in range(T):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = np.exp(g[0, t, 0]) * prev[0, 0, t]
        e = vt - St.T @ kt
        direction = np.outer(kt, e)
        loss = lambda a: 0.5 * np.sum(((St + a * direction).T @ kt - vt) ** 2)
        res = minimize_scalar(loss, bracket=(0.0, 1.0), tol=1e-12)
        dS = st[0, 0, t] - St
        alpha_oracle = np.sum(dS * direction) / np.sum(direction * direction)
        np.testing.assert_allclose(dS, alpha_oracle * direction, rtol=1e-9, atol=1e-12)
        assert abs(alpha_oracle - res.x) <= 1e-6 * abs(res.x), (alpha_oracle, res.x)


@pytest.mark.parametrize("eps", [0.0, 0.37])
def test_normalised_sgd_step(eps):
    """dS = -(eta/(||k||^2+eps)) * grad L(S~) with L(S) = 1/2||S^T k - v||^2,
    the gradient taken by autograd (independent of the oracle's arithmetic)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    B, T, H, dk, dv = 1, 8, 1, 7, 5
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=0.5)
    o, hT, st = oracle.kla_oracle_forward(q, k, v, g, eta, eps, h0, return_states=True)
    prev = _prev_states(st, h0, B, H, dk, dv)
    for t in range(T):
        kt, vt = k[0, t, 0], v[0, t, 0]
        St = np.exp(g[0, t, 0]) * prev[0, 0, t]
        S = torch.tensor(St, dtype=torch.float64, requires_grad=True)
        L = 0.5 * ((S.T @ torch.tensor(kt) - torch.tensor(vt)) ** 2).sum()
        (grad,) = torch.autograd.grad(L, S)
        step = -(eta[0, t, 0] / (kt @ kt + eps)) * grad.numpy()
        np.testing.assert_allclose(st[0, 0, t] - St, step, rtol=1e-10, atol=1e-13)


def test_relaxation_residual():
    """After the write, the residual shrinks by exactly 1 - eta||k||^2/(||k||^2+eps)."""
    rng = np.random.default_rng(15)
    B, T, H, dk, dv = 1, 16, 2, 8, 6
    eps = 0.21
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=0.4)
    o, hT, st = oracle.kla_oracle_forward(q, k, v, g, eta, eps, h0, return_states=True)
    prev = _prev_states(st, h0, B, H, dk, dv)
    for h in range(H):
        for t in range(T):
            kt, vt = k[0, t, h], v[0, t, h]
            St = np.exp(g[0, t, h]) * prev[0, h, t]
            e_before = vt - St.T @ kt
            e_after = vt - st[0, h, t].T @ kt
            shrink = 1.0 - eta[0, t, h] * (kt @ kt) / (kt @ kt + eps)
            np.testing.assert_allclose(e_after, shrink * e_before, rtol=1e-9, atol=1e-12)


def test_beta_zero_closed_form():
    """eta = 0 (beta = 0): the state only decays, o_t = exp(sum_{s<=t} g_s) h0^T q_t."""
    rng = np.random.default_rng(16)
    B, T, H, dk, dv = 2, 50, 3, 10, 6
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=1.0)
    eta = np.zeros_like(eta)
    o, hT = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    gam = np.cumsum(g, axis=1)  # [B,T,H]
    ref = np.exp(gam)[..., None] * np.einsum("bthi,bhij->bthj", q, h0)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT, np.exp(gam[:, -1])[..., None, None] * h0, rtol=1e-12)


@pytest.mark.parametrize("decay", [False, True])
def test_no_erase_equals_masked_attention(decay):
    """No-erase mode is plain (gated) linear attention; compare with the
    brute-force O(T^2) causal masked form
    o_t = sum_{s<=t} exp(gam_t - gam_s) (q_t . k_s) v_s + exp(gam_t) h0^T q_t."""
    rng = np.random.default_rng(17 + decay)
    B, T, H, dk, dv = 2, 33, 2, 5, 4
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=0.7)
    if not decay:
        g = np.zeros_like(g)
    o, hT = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0, no_erase=True)
    gam = np.cumsum(g, axis=1)
    ref = np.zeros_like(o)
    for b in range(B):
        for h in range(H):
            for t in range(T):
                acc = np.exp(gam[b, t, h]) * (q[b, t, h] @ h0[b, h])
                for s in range(t + 1):
                    acc = acc + np.exp(gam[b, t, h] - gam[b, s, h]) * (q[b, t, h] @ k[b, s, h]) * v[b, s, h]
                ref[b, t, h] = acc
    np.testing.assert_allclose(o, ref, rtol=1e-11, atol=1e-12)


def test_joint_key_value_scale_invariance_at_eps_zero():
    """With eps = 0 the constraint S^T k = v is homogeneous in (k, v), so
    rescaling k_t and v_t by the same per-token factor leaves the write
    beta_t k_t e_t^T, hence o and hT, unchanged (the key-norm normalisation
    of the coefficient)."""
    rng = np.random.default_rng(19)
    B, T, H, dk, dv = 1, 30, 2, 8, 8
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=0.2)
    o1, h1 = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0)
    scale = np.exp(rng.uniform(-2, 2, (B, T, H, 1)))
    o2, h2 = oracle.kla_oracle_forward(q, k * scale, v * scale, g, eta, 0.0, h0)
    np.testing.assert_allclose(o2, o1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(h2, h1, rtol=1e-10, atol=1e-12)


def test_threads_do_not_change_results():
    rng = np.random.default_rng(20)
    args = _rand_inputs(rng, 3, 20, 5, 8, 6, h0_std=0.1)
    o1, h1 = oracle.kla_oracle_forward(*args[:5], 1e-6, args[5], threads=1)
    o2, h2 = oracle.kla_oracle_forward(*args[:5], 1e-6, args[5], threads=7)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


def test_decode_steps_continue_the_forward():
    """T prefill tokens then n decode steps equal a prefill of T+n tokens."""
    rng = np.random.default_rng(21)
    B, T, H, dk, dv = 2, 9, 3, 6, 5
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, h0_std=0.3)
    o_full, h_full = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    o_pre, S = oracle.kla_oracle_forward(q[:, :5], k[:, :5], v[:, :5], g[:, :5], eta[:, :5], 1e-6, h0)
    np.testing.assert_array_equal(o_pre, o_full[:, :5])
    for t in range(5, T):
        ot, S = oracle.kla_oracle_decode_step(q[:, t], k[:, t], v[:, t], g[:, t], eta[:, t], 1e-6, S)
        np.testing.assert_allclose(ot, o_full[:, t], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(S, h_full, rtol=1e-13, atol=1e-14)


def test_empty_sequence_returns_h0():
    rng = np.random.default_rng(22)
    q, k, v, g, eta, h0 = _rand_inputs(rng, 1, 0, 2, 4, 3, h0_std=1.0)
    o, hT = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    assert o.shape == (1, 0, 2, 3)
    np.testing.assert_array_equal(hT, h0)


# ---- the direct step size beta_t = eta_t (the learned scalar of Gated
# DeltaNet that the page's sections "Problem statement" and "Methodology" say
# KLA replaces; with g = 0, the ungated delta rule)

def test_direct_beta_hand_worked_two_tokens():
    # d_k = 2, d_v = 1, h0 = 0.  Token 0: k = (1, 0), v = 2, q = (1, 1),
    # g = 0, eta = 0.5.  Token 1: k = (1, 1), v = 3, q = (0, 2), g = log 0.5,
    # eta = 0.25.
    #   direct:   S_1 = 0.5 * (1,0) * 2 = (1, 0);              o_0 = 1
    #             S~ = (0.5, 0), e = 3 - 0.5 = 2.5,
    #             S_2 = (0.5, 0) + 0.25 * (1,1) * 2.5 = (1.125, 0.625); o_1 = 1.25
    #   Kaczmarz (eps = 0): token 0 is the same (||k||^2 = 1); token 1 has
    #             beta = 0.25 / 2, S_2 = (0.8125, 0.3125), o_1 = 0.625
    q = np.array([[1.0, 1.0], [0.0, 2.0]]).reshape(1, 2, 1, 2)
    k = np.array([[1.0, 0.0], [1.0, 1.0]]).reshape(1, 2, 1, 2)
    v = np.array([2.0, 3.0]).reshape(1, 2, 1, 1)
    g = np.array([0.0, math.log(0.5)]).reshape(1, 2, 1)
    eta = np.array([0.5, 0.25]).reshape(1, 2, 1)
    o, hT = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, beta_direct=True)
    np.testing.assert_allclose(o.ravel(), [1.0, 1.25], rtol=0, atol=1e-15)
    np.testing.assert_allclose(hT.ravel(), [1.125, 0.625], rtol=0, atol=1e-15)
    o, hT = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0)
    np.testing.assert_allclose(o.ravel(), [1.0, 0.625], rtol=0, atol=1e-15)
    np.testing.assert_allclose(hT.ravel(), [0.8125, 0.3125], rtol=0, atol=1e-15)


def test_direct_beta_equals_kaczmarz_for_unit_keys():
    # ||k_t|| = 1 and eps = 0 make eta_t / (||k_t||^2 + eps) = eta_t
    rng = np.random.default_rng(31)
    q, k, v, g, eta, h0 = _rand_inputs(rng, 2, 40, 3, 8, 5, knorm=(1.0, 1.0), h0_std=0.3)
    o_d, h_d = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, beta_direct=True)
    o_k, h_k = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0)
    np.testing.assert_allclose(o_d, o_k, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h_d, h_k, rtol=1e-12, atol=1e-12)
    # and with other key norms the two differ
    q, k, v, g, eta, h0 = _rand_inputs(rng, 1, 40, 2, 8, 5, knorm=(2.0, 3.0))
    o_d, _ = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, beta_direct=True)
    o_k, _ = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0)
    assert np.max(np.abs(o_d - o_k)) > 1e-2


def test_delta_rule_projection_with_unit_keys():
    # g = 0, beta = 1, ||k|| = 1: the delta rule writes S_t^T k_t = v_t exactly
    rng = np.random.default_rng(32)
    B, T, H, dk, dv = 1, 30, 2, 6, 4
    q, k, v, _, _, h0 = _rand_inputs(rng, B, T, H, dk, dv, knorm=(1.0, 1.0), h0_std=0.5)
    g = np.zeros((B, T, H))
    eta = np.ones((B, T, H))
    _, _, states = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, beta_direct=True,
                                             return_states=True)
    for t in range(T):
        for h in range(H):
            np.testing.assert_allclose(states[0, h, t].T @ k[0, t, h], v[0, t, h], rtol=0, atol=1e-12)
