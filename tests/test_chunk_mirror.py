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
