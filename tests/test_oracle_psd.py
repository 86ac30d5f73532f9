"""Pins of the oracle's rank-one PSD feature map (DeltaKATA's keys and queries)."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("p", [1, 2, 5, 10, 15])
def test_feature_inner_product_is_squared_dot(p):
    # <psi(u), psi(w)>_F = (u . w)^2, the identity the KATA page builds on
    rng = np.random.default_rng(p)
    u, w = rng.standard_normal((2, 7, p))
    d = 128 if p > 10 else 64
    yu, yw = oracle.kla_oracle_psd_features(u, d), oracle.kla_oracle_psd_features(w, d)
    assert np.allclose((yu * yw).sum(-1), (u * w).sum(-1) ** 2, rtol=1e-12, atol=1e-12)
    # the norm of a feature is the squared norm of its vector
    assert np.allclose(np.linalg.norm(yu, axis=-1), (u * u).sum(-1), rtol=1e-12)


def test_feature_is_the_outer_product():
    # unpacking the vector gives numpy's outer product u u^T
    rng = np.random.default_rng(3)
    u = rng.standard_normal(6)
    y = oracle.kla_oracle_psd_features(u, 64)
    M = np.zeros((6, 6))
    for n, (i, j) in enumerate(oracle.psd_feature_index(6)):
        v = y[n] if i == j else y[n] / np.sqrt(2.0)
        M[i, j] = M[j, i] = v
    assert np.allclose(M, np.outer(u, u), rtol=1e-14, atol=1e-14)
    assert np.all(y[21:] == 0.0)   # zero padding past p(p+1)/2 = 21


def test_feature_backward_matches_finite_differences():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 15))
    dy = rng.standard_normal((3, 128))
    got = oracle.kla_oracle_psd_features_bwd(x, dy)
    h = 1e-6
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        num[idx] = ((oracle.kla_oracle_psd_features(xp, 128) - oracle.kla_oracle_psd_features(xm, 128))
                    * dy).sum() / (2 * h)
    assert np.abs(got - num).max() < 1e-7 * max(1.0, np.abs(num).max())


def test_deltakata_step_size_uses_the_fourth_power():
    # the Kaczmarz step on features divides by ||psi(k)||^2 = ||k||^4: with
    # eta = 1, eps = 0 and no decay, S_1^T psi(k) = v exactly
    rng = np.random.default_rng(9)
    k = rng.standard_normal((1, 1, 1, 15)) * 1.3
    q = rng.standard_normal((1, 1, 1, 15))
    v = rng.standard_normal((1, 1, 1, 4))
    fk = oracle.kla_oracle_psd_features(k, 128)
    fq = oracle.kla_oracle_psd_features(q, 128)
    g = np.zeros((1, 1, 1))
    eta = np.ones((1, 1, 1))
    o, hT = oracle.kla_oracle_forward(fq, fk, v, g, eta, 0.0)
    assert np.allclose(hT[0, 0].T @ fk[0, 0, 0], v[0, 0, 0], rtol=1e-12)
    # from a zero state: o = (psi(q) . psi(k)) v / ||k||^4 = (q . k)^2 v / ||k||^4
    qk = (q * k).sum()
    assert np.allclose(o[0, 0, 0], qk ** 2 * v[0, 0, 0] / (k * k).sum() ** 2, rtol=1e-12)
