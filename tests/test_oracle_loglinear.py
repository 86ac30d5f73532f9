"""Pins of the oracle's Log-Linear gated delta rule."""
import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _rand_inputs


def _fenwick_buckets(t):
    """The prefix 0..t split the Fenwick way, built without the level formula:
    peel off aligned blocks from t downwards; block sizes 1, then 2^b for each
    set bit b of t, smallest first.  Returns {level: tokens}."""
    buckets = {0: [t]}
    end = t                      # tokens below `end` are still unassigned
    for b in range(t.bit_length()):
        if (t >> b) & 1:
            start = end - (1 << b)
            buckets[b + 1] = list(range(start, end))
            end = start
    assert end == 0
    return buckets


@pytest.mark.parametrize("t", list(range(0, 70)) + [255, 256, 1000, 4095])
def test_level_function_is_the_fenwick_partition(t):
    for lev, toks in _fenwick_buckets(t).items():
        for s in toks:
            assert oracle.loglinear_level(t, s) == lev
        assert len(toks) == (1 if lev == 0 else 1 << (lev - 1))


def test_number_of_levels():
    assert [oracle.loglinear_num_levels(T) for T in (1, 2, 3, 4, 5, 64, 65, 4096, 4097)] == \
        [1, 2, 3, 3, 4, 7, 8, 13, 14]
    for T in (2, 3, 17, 64, 65, 300):
        assert max(oracle.loglinear_level(T - 1, s) for s in range(T)) < oracle.loglinear_num_levels(T)


@pytest.mark.parametrize("direct", [False, True])
def test_unit_weights_give_the_ordinary_recurrence(direct):
    rng = np.random.default_rng(11)
    q, k, v, g, eta, _ = _rand_inputs(rng, 2, 37, 2, 5, 3, knorm=(0.5, 1.5))
    L = oracle.loglinear_num_levels(37)
    lam = np.ones((2, 37, 2, L))
    o = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 0.1, beta_direct=direct)
    o_ref, _ = oracle.kla_oracle_forward(q, k, v, g, eta, 0.1, beta_direct=direct)
    assert np.allclose(o, o_ref, rtol=1e-11, atol=1e-12)


def test_level_zero_alone_is_the_token_itself():
    # lambda = e_0: o_t = beta_t (q_t . k_t) v_t
    rng = np.random.default_rng(12)
    q, k, v, g, eta, _ = _rand_inputs(rng, 1, 20, 1, 4, 3)
    lam = np.zeros((1, 20, 1, oracle.loglinear_num_levels(20)))
    lam[..., 0] = 1.0
    eps = 0.05
    o = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, eps)
    beta = eta / ((k * k).sum(-1) + eps)
    want = (beta * (q * k).sum(-1))[..., None] * v
    assert np.allclose(o, want, rtol=1e-12)


def test_linear_attention_case_is_the_hierarchical_mask():
    # without the erase term: O = (Q K^T o M_H) V with M_H[t, s] = lambda_t^(level) exp(sum g_{s+1..t})
    rng = np.random.default_rng(13)
    T = 45
    q, k, v, g, eta, _ = _rand_inputs(rng, 1, T, 1, 4, 3)
    lam = rng.uniform(0.2, 1.5, (1, T, 1, oracle.loglinear_num_levels(T)))
    o = oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 0.0, no_erase=True)
    cg = np.cumsum(g[0, :, 0])
    M = np.zeros((T, T))
    for t in range(T):
        for s in range(t + 1):
            M[t, s] = lam[0, t, 0, oracle.loglinear_level(t, s)] * np.exp(cg[t] - cg[s])
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    assert np.allclose(o[0, :, 0], ((Q @ K.T) * M) @ V, rtol=1e-11, atol=1e-12)


def test_buckets_split_the_state():
    # sum over one-hot weights equals unit weights (linearity in lambda)
    rng = np.random.default_rng(14)
    T = 30
    q, k, v, g, eta, _ = _rand_inputs(rng, 1, T, 1, 3, 2)
    L = oracle.loglinear_num_levels(T)
    total = 0
    for lev in range(L):
        lam = np.zeros((1, T, 1, L))
        lam[..., lev] = 1.0
        total = total + oracle.kla_oracle_loglinear_forward(q, k, v, g, eta, lam, 0.1)
    o_ref, _ = oracle.kla_oracle_forward(q, k, v, g, eta, 0.1)
    assert np.allclose(total, o_ref, rtol=1e-11, atol=1e-12)
