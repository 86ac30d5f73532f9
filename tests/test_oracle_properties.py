"""Property tests of the fp64 oracle over random small shapes (Hypothesis).

Each property follows from the recurrence of "KLA: Kaczmarz Linear
Attention", section "KLA update rule", for any inputs:
  - for fixed keys and gates the map (V, h0) -> (o, hT) is linear: the update
    S_t = a_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T is affine in
    S and linear in v, and o_t = S_t^T q_t is linear in S_t and in q_t;
  - heads and batch entries are independent: permuting them permutes the
    outputs;
  - splitting the sequence and carrying the state equals one call;
  - the chunked form (any chunk length) equals the sequential one;
  - at eta = 1, eps = 0 every step satisfies S_t^T k_t = v_t.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import chunk_mirror as cm

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SHAPES = st.tuples(st.integers(1, 2), st.integers(0, 40), st.integers(1, 3), st.integers(1, 6),
                   st.integers(1, 5))
SEEDS = st.integers(0, 2**31 - 1)


def _inputs(seed, B, T, H, dk, dv, knorm=(0.25, 4.0), projection=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, H, dk))
    u = rng.standard_normal((B, T, H, dk))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    k = u * np.exp(rng.uniform(math.log(knorm[0]), math.log(knorm[1]), (B, T, H, 1)))
    v = rng.standard_normal((B, T, H, dv))
    if projection:
        g, eta = np.zeros((B, T, H)), np.ones((B, T, H))
    else:
        g = -np.log1p(np.exp(-(rng.standard_normal((B, T, H)) + 2.0)))
        eta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    h0 = rng.standard_normal((B, H, dk, dv)) * 0.5
    return q, k, v, g, eta, h0


def _close(a, b, tol=1e-10):
    scale = max(np.abs(b).max(), 1.0) if b.size else 1.0
    return a.shape == b.shape and (a.size == 0 or np.abs(a - b).max() <= tol * scale)


@settings(max_examples=40, deadline=None)
@given(SHAPES, SEEDS, st.floats(-3.0, 3.0), st.floats(-3.0, 3.0))
def test_linear_in_values_and_start_state(shape, seed, alpha, gamma):
    B, T, H, dk, dv = shape
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv)
    _, _, v2, _, _, h02 = _inputs(seed + 1, B, T, H, dk, dv)
    o1, s1 = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    o2, s2 = oracle.kla_oracle_forward(q, k, v2, g, eta, 1e-6, h02)
    o3, s3 = oracle.kla_oracle_forward(q, k, alpha * v + gamma * v2, g, eta, 1e-6, alpha * h0 + gamma * h02)
    assert _close(o3, alpha * o1 + gamma * o2)
    assert _close(s3, alpha * s1 + gamma * s2)


@settings(max_examples=30, deadline=None)
@given(SHAPES, SEEDS, st.floats(-2.0, 2.0))
def test_linear_in_queries(shape, seed, alpha):
    B, T, H, dk, dv = shape
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv)
    o1, s1 = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    o2, s2 = oracle.kla_oracle_forward(alpha * q, k, v, g, eta, 1e-6, h0)
    assert _close(o2, alpha * o1)
    assert _close(s2, s1, 0.0)


@settings(max_examples=30, deadline=None)
@given(SHAPES, SEEDS, st.randoms(use_true_random=False))
def test_permuting_heads_and_batch_permutes_outputs(shape, seed, rnd):
    B, T, H, dk, dv = shape
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv)
    pb = list(range(B))
    ph = list(range(H))
    rnd.shuffle(pb)
    rnd.shuffle(ph)
    o, s = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    perm = lambda x: x[pb][:, :, ph] if x.ndim == 4 and x.shape[1] == T else x[pb][:, ph]  # noqa: E731
    o2, s2 = oracle.kla_oracle_forward(perm(q), perm(k), perm(v), g[pb][:, :, ph], eta[pb][:, :, ph], 1e-6,
                                       h0[pb][:, ph])
    assert _close(o2, o[pb][:, :, ph], 0.0)
    assert _close(s2, s[pb][:, ph], 0.0)


@settings(max_examples=30, deadline=None)
@given(SHAPES, SEEDS, st.integers(0, 40))
def test_split_sequence_carries_the_state(shape, seed, cut):
    B, T, H, dk, dv = shape
    cut = min(cut, T)
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv)
    o, s = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0)
    oa, sa = oracle.kla_oracle_forward(q[:, :cut], k[:, :cut], v[:, :cut], g[:, :cut], eta[:, :cut], 1e-6, h0)
    ob, sb = oracle.kla_oracle_forward(q[:, cut:], k[:, cut:], v[:, cut:], g[:, cut:], eta[:, cut:], 1e-6, sa)
    assert _close(np.concatenate([oa, ob], axis=1), o, 1e-12)
    assert _close(sb, s, 1e-12)


@settings(max_examples=30, deadline=None)
@given(SHAPES, SEEDS, st.integers(1, 45), st.booleans())
def test_chunked_form_equals_the_sequential_loop(shape, seed, C, direct):
    B, T, H, dk, dv = shape
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv, knorm=(0.5, 1.2) if direct else (0.25, 4.0))
    o, s = oracle.kla_oracle_forward(q, k, v, g, eta, 1e-6, h0, beta_direct=direct)
    oc, sc = cm.chunk_forward(q, k, v, g, eta, 1e-6, h0, C=C, beta_direct=direct)
    assert _close(oc, o, 1e-11)
    assert _close(sc, s, 1e-11)


@settings(max_examples=30, deadline=None)
@given(st.tuples(st.integers(1, 2), st.integers(1, 30), st.integers(1, 2), st.integers(2, 8),
                 st.integers(1, 4)), SEEDS)
def test_projection_constraint_every_step(shape, seed):
    B, T, H, dk, dv = shape
    T = min(T, dk)   # keys of one sequence stay independent enough for a clean check
    q, k, v, g, eta, h0 = _inputs(seed, B, T, H, dk, dv, knorm=(0.5, 2.0), projection=True)
    _, _, states = oracle.kla_oracle_forward(q, k, v, g, eta, 0.0, h0, return_states=True)
    resid = np.einsum("bhtkv,bthk->bthv", states, k) - v
    assert np.abs(resid).max() <= 1e-9 * max(1.0, np.abs(v).max())
