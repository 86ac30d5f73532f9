"""Pins of the oracle's reverse mode (``oracle.kla_oracle_backward``).

The derivative is checked against things other than itself:
- central finite differences of ``kla_oracle_forward`` (the forward is pinned
  on its own in ``test_oracle_pins``);
- torch autograd through a plain fp64 loop of the recurrence;
- the closed form at eta = 0, where the state only decays;
- planted mistakes in a copy of the C source, each caught by the
  finite-difference pin.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests.test_oracle_pins import _rand_inputs

SRC = os.path.join(os.path.dirname(oracle.__file__), "kla_oracle.c")
NAMES = ("q", "k", "v", "g", "eta", "h0")


def _loss(inp, dout, dhT, eps, direct):
    o, hT = oracle.kla_oracle_forward(*(inp[n] for n in NAMES[:5]), eps, inp["h0"],
                                      beta_direct=direct)
    return float((o * dout).sum() + (hT * dhT).sum())


def _case(seed, B=1, T=6, H=2, dk=3, dv=2, knorm=(0.5, 2.0)):
    rng = np.random.default_rng(seed)
    q, k, v, g, eta, h0 = _rand_inputs(rng, B, T, H, dk, dv, knorm=knorm, h0_std=0.5)
    inp = dict(q=q, k=k, v=v, g=g, eta=eta, h0=h0)
    dout = rng.standard_normal(v.shape)
    dhT = rng.standard_normal(h0.shape)
    return inp, dout, dhT


def _finite_difference_check(inp, dout, dhT, eps, direct, tol=1e-6):
    grads = oracle.kla_oracle_backward(*(inp[n] for n in NAMES[:5]), eps, inp["h0"], dout, dhT,
                                       beta_direct=direct)
    h = 1e-6
    for name in NAMES:
        x = inp[name]
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + h
            lp = _loss(inp, dout, dhT, eps, direct)
            x[idx] = keep - h
            lm = _loss(inp, dout, dhT, eps, direct)
            x[idx] = keep
            num[idx] = (lp - lm) / (2 * h)
        got = grads["d" + name]
        scale = max(1.0, np.abs(num).max())
        err = np.abs(got - num).max() / scale
        assert err < tol, f"d{name}: max err {err:.3e} (direct={direct}, eps={eps})"


@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_backward_matches_finite_differences(direct, eps):
    inp, dout, dhT = _case(7 + int(direct) + int(eps * 10))
    _finite_difference_check(inp, dout, dhT, eps, direct)


def test_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    inp, dout, dhT = _case(21, B=2, T=20, H=2, dk=4, dv=3)
    eps = 0.05
    t = {n: torch.tensor(inp[n], dtype=torch.float64, requires_grad=True) for n in NAMES}
    B, T, H, dk = inp["k"].shape
    outs = []
    S = t["h0"]
    for s in range(T):
        k = t["k"][:, s]                                  # [B,H,dk]
        beta = t["eta"][:, s] / ((k * k).sum(-1) + eps)    # [B,H]
        St = torch.exp(t["g"][:, s])[..., None, None] * S
        e = t["v"][:, s] - torch.einsum("bhij,bhi->bhj", St, k)
        S = St + beta[..., None, None] * k[..., :, None] * e[..., None, :]
        outs.append(torch.einsum("bhij,bhi->bhj", S, t["q"][:, s]))
    o = torch.stack(outs, 1)
    loss = (o * torch.tensor(dout)).sum() + (S * torch.tensor(dhT)).sum()
    loss.backward()
    grads = oracle.kla_oracle_backward(*(inp[n] for n in NAMES[:5]), eps, inp["h0"], dout, dhT)
    for n in NAMES:
        ref = t[n].grad.numpy()
        assert np.abs(grads["d" + n] - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max()), n


def test_backward_closed_form_at_zero_step():
    # eta = 0: S_t = Gamma_t h0 with Gamma_t = exp(sum_{s<=t} g_s), o_t = Gamma_t h0^T q_t
    inp, dout, dhT = _case(33, B=1, T=7, H=1, dk=3, dv=4)
    inp["eta"][:] = 0.0
    eps = 0.2
    grads = oracle.kla_oracle_backward(*(inp[n] for n in NAMES[:5]), eps, inp["h0"], dout, dhT)
    q, k, v, g, h0 = (inp[n][0, :, 0] if n != "h0" else inp[n][0, 0] for n in ("q", "k", "v", "g", "h0"))
    do, dh = dout[0, :, 0], dhT[0, 0]
    Gam = np.exp(np.cumsum(g))
    T = len(g)
    # dq_t = Gamma_t h0 do_t
    assert np.allclose(grads["dq"][0, :, 0], Gam[:, None] * (do @ h0.T), atol=1e-12)
    # dh0 = sum_t Gamma_t q_t do_t^T + Gamma_T dhT
    assert np.allclose(grads["dh0"][0, 0], np.einsum("t,ti,tj->ij", Gam, q, do) + Gam[-1] * dh,
                       atol=1e-12)
    # dg_s = sum_{t>=s} do_t . o_t + <dhT, Gamma_T h0>
    per_t = Gam * np.einsum("ti,ij,tj->t", q, h0, do)
    want_dg = np.cumsum(per_t[::-1])[::-1] + Gam[-1] * (dh * h0).sum()
    assert np.allclose(grads["dg"][0, :, 0], want_dg, atol=1e-12)
    # k and v have no influence at beta = 0
    assert np.abs(grads["dk"]).max() == 0.0 and np.abs(grads["dv"]).max() == 0.0
    # deta_t = k_t^T dS_t e_t / (||k_t||^2 + eps), dS_t = sum_{t'>=t} (Gamma_t'/Gamma_t) q_t' do_t'^T
    #          + (Gamma_T/Gamma_t) dhT, e_t = v_t - Gamma_t h0^T k_t
    for t in range(T):
        dS = sum(Gam[u] / Gam[t] * np.outer(q[u], do[u]) for u in range(t, T)) + Gam[-1] / Gam[t] * dh
        e = v[t] - Gam[t] * h0.T @ k[t]
        want = k[t] @ dS @ e / (k[t] @ k[t] + eps)
        assert abs(grads["deta"][0, t, 0] - want) <= 1e-12 * max(1.0, abs(want))


def test_backward_empty_and_shapes():
    inp, dout, dhT = _case(41, T=0)
    grads = oracle.kla_oracle_backward(*(inp[n] for n in NAMES[:5]), 1e-6, inp["h0"], dout, dhT)
    assert np.array_equal(grads["dh0"], dhT)   # nothing happens between h0 and hT
    assert grads["dq"].shape == inp["q"].shape and grads["dg"].shape == inp["g"].shape


BWD_MUTATIONS = {
    "readout_term_dropped": ("dS[i * dv + j] += qt[i] * dot[j];", "dS[i * dv + j] += 0.0 * dot[j];"),
    "dq_from_previous_state": ("acc += S[i * dv + j] * dot[j];", "acc += Sp[i * dv + j] * dot[j];"),
    "residual_sign": ("dS[i * dv + j] -= kt[i] * de[j];", "dS[i * dv + j] += kt[i] * de[j];"),
    "decay_gradient_without_gate": ("J->dg[tok] = a * da;", "J->dg[tok] = da;"),
    "step_size_chain_dropped": ("dkt[i] -= 2.0 * beta * dbeta / den * kt[i];", "dkt[i] -= 0.0;"),
    "key_residual_term_dropped": ("dkt[i] -= r;", "dkt[i] -= 0.0 * r;"),
    "state_not_decayed": ("dS[i] *= a;", "dS[i] *= 1.0;"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTATIONS))
def test_backward_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = BWD_MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    mutated = tmp_path / "kla_oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(mutated), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    real = oracle._load()
    for fn in ("kla_oracle_forward", "kla_oracle_backward"):
        getattr(lib, fn).argtypes = getattr(real, fn).argtypes
        getattr(lib, fn).restype = ctypes.c_int
    monkeypatch.setattr(oracle, "_lib", lib)
    inp, dout, dhT = _case(55)
    with pytest.raises(AssertionError):
        _finite_difference_check(inp, dout, dhT, 0.3, False)
