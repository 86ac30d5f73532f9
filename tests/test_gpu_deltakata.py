"""GPU parity of DeltaKATA: the PSD feature map (forward and derivative) and
the KLA recurrence run on those features, against the oracle."""
import numpy as np
import pytest
import torch

import kla_inputs
import oracle
from tests.parity_utils import TOL, rel_err

pytestmark = pytest.mark.gpu


def _kla():
    import chunked_delta_rule_kla_gb300 as kla
    return kla


def _dt(io):
    return torch.bfloat16 if io == "bf16" else torch.float32


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("p,d", [(1, 64), (4, 64), (10, 64), (10, 128), (15, 128)])
def test_features_match_oracle(io, p, d):
    kla = _kla()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(p * 7 + d)
    x = torch.randn((3, 37, 2, p), generator=gen, device="cuda").to(_dt(io))
    y = kla.psd_features(x, d)
    torch.cuda.synchronize()
    ref = oracle.kla_oracle_psd_features(x, d)
    # fp32 products of the stored inputs, rounded once to the I/O dtype
    ulp = 2.0 ** -8 if io == "bf16" else 2.0 ** -21
    err = np.abs(y.double().cpu().numpy() - ref)
    assert np.all(err <= ulp * np.abs(ref) + 1e-30), err.max()
    assert bool((y[..., p * (p + 1) // 2:].float() == 0).all())


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("p,d", [(3, 64), (15, 128)])
def test_feature_derivative_matches_oracle(io, p, d):
    kla = _kla()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(100 + p)
    x = torch.randn((4, 50, 3, p), generator=gen, device="cuda").to(_dt(io))
    gy = torch.randn((4, 50, 3, d), generator=gen, device="cuda").to(_dt(io))
    gx = torch.empty_like(x)
    kla.kla_psd_features_bwd(x, gy, gx)
    torch.cuda.synchronize()
    ref = oracle.kla_oracle_psd_features_bwd(x, gy)
    assert rel_err(gx, ref) <= TOL[io]


def _case(io, p, dv, T=130, seed=500):
    case = kla_inputs.TINY.with_(B=2, T=T, H=2, dk=p, dv=dv, io=io, h0_std=0.05, seed=seed,
                                 knorm=(0.6, 1.6))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    B, H = case.B, case.H
    dt = _dt(io)
    q = torch.randn((B, T, H, p), generator=gen, device="cuda").mul(0.4).to(dt)
    u = torch.randn((B, T, H, p), generator=gen, device="cuda")
    k = (u / u.norm(dim=-1, keepdim=True) * torch.empty((B, T, H, 1), device="cuda").uniform_(
        0.6, 1.6, generator=gen)).to(dt)
    v = torch.randn((B, T, H, dv), generator=gen, device="cuda").to(dt)
    g = torch.nn.functional.logsigmoid(torch.randn((B, T, H), generator=gen, device="cuda") + 2.0)
    eta = torch.sigmoid(torch.randn((B, T, H), generator=gen, device="cuda"))
    h0 = torch.randn((B, H, 128 if p > 10 else 64, dv), generator=gen, device="cuda") * 0.05
    return q, k, v, g, eta, h0


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("p,dv", [(15, 128), (10, 64)])
def test_recurrence_on_gpu_features(io, p, dv):
    # the chunked forward on the features the GPU made, against the oracle on the same values
    kla = _kla()
    q, k, v, g, eta, h0 = _case(io, p, dv)
    d = 128 if p > 10 else 64
    fq, fk = kla.psd_features(q, d), kla.psd_features(k, d)
    o, hT = kla.chunk_fwd(fq, fk, v, g, eta, 1e-6, h0)
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.kla_oracle_forward(fq, fk, v, g, eta, 1e-6, h0)
    assert rel_err(o, o_ref) <= TOL[io]
    assert rel_err(hT, h_ref) <= TOL[io]


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_deltakata_end_to_end_forward_and_backward(io):
    # from raw q, k: features, recurrence and their derivatives, through autograd
    kla = _kla()
    p, dv = 15, 128
    q, k, v, g, eta, h0 = _case(io, p, dv, T=150, seed=510)
    leaves = {n: t.clone().requires_grad_(True) for n, t in
              dict(q=q, k=k, v=v, g=g, eta=eta, h0=h0).items()}
    o, hT = kla.deltakata(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["eta"], 1e-6,
                          leaves["h0"])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(520)
    do = torch.randn(o.shape, generator=gen, device="cuda").to(o.dtype)
    dh = torch.randn(hT.shape, generator=gen, device="cuda")
    (o.float() * do.float()).sum().add_((hT * dh).sum()).backward()
    torch.cuda.synchronize()
    fq, fk = oracle.kla_oracle_psd_features(q, 128), oracle.kla_oracle_psd_features(k, 128)
    o_ref, h_ref = oracle.kla_oracle_forward(fq, fk, v, g, eta, 1e-6, h0)
    assert rel_err(o, o_ref) <= TOL[io]
    assert rel_err(hT, h_ref) <= TOL[io]
    gr = oracle.kla_oracle_backward(fq, fk, v, g, eta, 1e-6, h0, do, dh)
    want = dict(q=oracle.kla_oracle_psd_features_bwd(q, gr["dq"]),
                k=oracle.kla_oracle_psd_features_bwd(k, gr["dk"]),
                v=gr["dv"], g=gr["dg"], eta=gr["deta"], h0=gr["dh0"])
    for n, leaf in leaves.items():
        e = rel_err(leaf.grad, want[n])
        assert e <= TOL[io], f"d{n}: {e:.3e}"


def _fused_vs_features(B, T, H, p, seed, h0=False, beta=0):
    """kla_deltakata_fwd (features formed inside the prefill) against
    kla_psd_features + kla_chunk_fwd_ex on the same inputs."""
    kla = _kla()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    dt = torch.bfloat16
    q = torch.randn((B, T, H, p), generator=gen, device="cuda").mul(0.4).to(dt)
    u = torch.randn((B, T, H, p), generator=gen, device="cuda")
    k = (u / u.norm(dim=-1, keepdim=True) * torch.empty((B, T, H, 1), device="cuda").uniform_(
        0.5, 2.0, generator=gen)).to(dt)
    v = torch.randn((B, T, H, 128), generator=gen, device="cuda").to(dt)
    g = torch.nn.functional.logsigmoid(torch.randn((B, T, H), generator=gen, device="cuda") + 2.0)
    eta = torch.sigmoid(torch.randn((B, T, H), generator=gen, device="cuda"))
    s0 = torch.randn((B, H, 128, 128), generator=gen, device="cuda") * 0.05 if h0 else None
    n = kla.kla_deltakata_fwd_workspace_bytes(B, T, H, p, 128)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    o = torch.empty((B, T, H, 128), dtype=dt, device="cuda")
    hT = torch.empty((B, H, 128, 128), dtype=torch.float32, device="cuda")
    kla.kla_deltakata_fwd(q, k, v, g, eta, 1e-6, s0, o, hT, ws, beta=beta)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK
    fq, fk = kla.psd_features(q, 128), kla.psd_features(k, 128)
    o2 = torch.empty_like(o)
    h2 = torch.empty_like(hT)
    ws2 = kla.alloc_workspace(B, T, H, 128, 128, 64, kla.KLA_IO_BF16, q.device)
    kla.kla_chunk_fwd_ex(fq, fk, v, g, eta, 1e-6, s0, o2, h2, ws2, beta=beta)
    torch.cuda.synchronize()
    return (q, k, v, g, eta, s0), (o, hT), (o2, h2)


@pytest.mark.parametrize("B,T,H,p,h0,beta", [
    (1, 300, 2, 15, False, 0),     # ragged last chunk, fused grid
    (2, 1000, 3, 11, True, 0),     # start state
    (1, 64, 1, 1, False, 0),       # one value per token, one chunk
    (3, 129, 5, 12, True, 1),      # direct step size, a one-token chunk
    (1, 2100, 40, 15, False, 0),   # 40 heads of 33 chunks (fused grid, no scan)
    (1, 128, 140, 15, True, 0),    # 140 heads: the prep grid and one carry grid
])
def test_fused_features_equal_features_then_prefill(B, T, H, p, h0, beta):
    # the same feature bytes reach the same kernels: o and hT agree bit for bit
    _, (o, hT), (o2, h2) = _fused_vs_features(B, T, H, p, 700 + 13 * p + H, h0, beta)
    assert torch.equal(o, o2)
    assert torch.equal(hT, h2)


def test_fused_forward_matches_oracle():
    # and against the oracle directly (features and recurrence in fp64)
    (q, k, v, g, eta, s0), (o, hT), _ = _fused_vs_features(2, 200, 2, 15, 790, True)
    fq, fk = oracle.kla_oracle_psd_features(q, 128), oracle.kla_oracle_psd_features(k, 128)
    o_ref, h_ref = oracle.kla_oracle_forward(fq, fk, v, g, eta, 1e-6, s0)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


@pytest.mark.parametrize("B,T,H,p,h0", [
    (1, 4096, 2, 15, True),      # two heads: the chunk-level scan (2 runs), a start state
    (1, 2100, 100, 12, False),   # 100 heads of 33 chunks: chunk ranges
])
def test_fused_features_on_the_scan_and_range_paths(B, T, H, p, h0):
    kla = _kla()
    assert kla.kla_chunk_fwd_auto_segments(B, T, H, 128, 128) == (2 if H == 2 else 1)
    _, (o, hT), (o2, h2) = _fused_vs_features(B, T, H, p, 900 + H, h0)
    assert torch.equal(o, o2)
    assert torch.equal(hT, h2)
