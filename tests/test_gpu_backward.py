"""GPU parity of the chunkwise backward (kla_chunk_bwd) against the oracle's
fp64 reverse mode, gradient by gradient, on the same seeded inputs."""
import pytest
import torch

import kla_inputs
import oracle
from tests.parity_utils import TOL, rel_err

pytestmark = pytest.mark.gpu

GRADS = ("dq", "dk", "dv", "dg", "deta", "dh0")


def _kla():
    import chunked_delta_rule_kla_gb300 as kla
    return kla


def _grad_inputs(inp, seed, dhT=True):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    B, T, H, dv = inp["v"].shape
    dk = inp["k"].shape[-1]
    do = torch.randn((B, T, H, dv), generator=gen, device="cuda").to(inp["q"].dtype)
    dh = torch.randn((B, H, dk, dv), generator=gen, device="cuda") if dhT else None
    return do, dh


def _check(inp, io, do, dhT, direct=False, heads=None, tol=None):
    kla = _kla()
    beta = kla.KLA_BETA_DIRECT if direct else kla.KLA_BETA_KACZMARZ
    got = kla.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], do, dhT, inp["eps"],
                        inp["h0"], beta=beta)
    torch.cuda.synchronize()
    sel = {}
    names = ("q", "k", "v", "g", "eta")
    if heads is not None:
        idx = torch.as_tensor(heads, device="cuda")
        sel = {n: inp[n].index_select(2, idx) for n in names}
        h0 = inp["h0"].index_select(1, idx) if inp["h0"] is not None else None
        do_s = do.index_select(2, idx)
        dh_s = dhT.index_select(1, idx) if dhT is not None else None
        got = {n: (t.index_select(1, idx) if n == "dh0" else t.index_select(2, idx))
               for n, t in got.items()}
    else:
        sel = {n: inp[n] for n in names}
        h0, do_s, dh_s = inp["h0"], do, dhT
    ref = oracle.kla_oracle_backward(*(sel[n] for n in names), inp["eps"], h0, do_s, dh_s,
                                     beta_direct=direct)
    tol = TOL[io] if tol is None else tol
    for n in GRADS:
        e = rel_err(got[n], ref[n])
        assert e <= tol, f"{n}: rel err {e:.3e} > {tol}"
    return got


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 130, 257])
def test_backward_ragged_lengths(io, T):
    case = kla_inputs.TINY.with_(B=2, T=T, H=2, dk=128, dv=128, io=io, h0_std=0.05, seed=300 + T)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 400 + T)
    _check(inp, io, do, dh)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_backward_head_dims(dk, dv, io):
    case = kla_inputs.TINY.with_(B=1, T=200, H=3, dk=dk, dv=dv, io=io, h0_std=0.05, seed=310 + dk + dv)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 410 + dk + dv)
    _check(inp, io, do, dh)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_backward_without_h0_and_dhT(io):
    case = kla_inputs.TINY.with_(B=2, T=150, H=2, dk=128, dv=128, io=io, h0_std=0.0, seed=320)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, _ = _grad_inputs(inp, 420, dhT=False)
    _check(inp, io, do, None)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_backward_direct_step_size(io):
    case = kla_inputs.TINY.with_(B=2, T=190, H=2, dk=128, dv=128, io=io, h0_std=0.05,
                                 knorm=(0.5, 1.2), seed=330)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 430)
    _check(inp, io, do, dh, direct=True)


def test_backward_deltanet_without_decay():
    case = kla_inputs.TINY.with_(B=1, T=160, H=2, dk=128, dv=128, io="bf16", h0_std=0.05,
                                 knorm=(0.5, 1.2), seed=340)
    inp = kla_inputs.make_prefill(case, device="cuda")
    inp["g"] = torch.zeros_like(inp["g"])
    do, dh = _grad_inputs(inp, 440)
    _check(inp, "bf16", do, dh, direct=True)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_backward_strong_decay(io):
    # log-decays near -3 per token: spans of about 190 inside a chunk
    case = kla_inputs.TINY.with_(B=1, T=130, H=2, dk=128, dv=128, io=io, h0_std=0.05, seed=350)
    inp = kla_inputs.make_prefill(case, device="cuda")
    inp["g"] = torch.full_like(inp["g"], -3.0)
    do, dh = _grad_inputs(inp, 450)
    _check(inp, io, do, dh)


def test_backward_odd_batch_and_heads():
    # B = 3, H = 3 with d_k = d_v = 128 in bf16 (the tensor-core kernels): token
    # rows interleave three heads, and the carries' grid has 18 CTAs
    case = kla_inputs.TINY.with_(B=3, T=190, H=3, dk=128, dv=128, io="bf16", h0_std=0.05, seed=365)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 465)
    _check(inp, "bf16", do, dh)


def test_backward_large_start_state():
    # h0 of unit scale: the residual e = v - Gam k S0 - ... is dominated by the
    # start state, the case that needs S0 at fp32-level accuracy in the products
    case = kla_inputs.TINY.with_(B=1, T=200, H=2, dk=128, dv=128, io="bf16", h0_std=1.0, seed=360)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 460)
    _check(inp, "bf16", do, dh)


def test_backward_empty_sequence():
    kla = _kla()
    case = kla_inputs.TINY.with_(B=1, T=0, H=2, dk=128, dv=128, io="bf16", h0_std=0.05, seed=360)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 460)
    got = kla.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], do, dh, inp["eps"],
                        inp["h0"])
    torch.cuda.synchronize()
    assert torch.equal(got["dh0"], dh)


def test_autograd_function_matches_oracle():
    kla = _kla()
    case = kla_inputs.TINY.with_(B=2, T=100, H=2, dk=128, dv=128, io="bf16", h0_std=0.05, seed=370)
    inp = kla_inputs.make_prefill(case, device="cuda")
    do, dh = _grad_inputs(inp, 470)
    leaves = {n: inp[n].clone().requires_grad_(True) for n in ("q", "k", "v", "g", "eta", "h0")}
    o, hT = kla.kla_chunk(*(leaves[n] for n in ("q", "k", "v", "g", "eta")), inp["eps"], leaves["h0"])
    (o.float() * do.float()).sum().add_((hT * dh).sum()).backward()
    ref = oracle.kla_oracle_backward(*(inp[n] for n in ("q", "k", "v", "g", "eta")), inp["eps"],
                                     inp["h0"], do, dh)
    for n, leaf in leaves.items():
        e = rel_err(leaf.grad, ref["d" + n])
        assert e <= TOL["bf16"], f"d{n}: {e:.3e}"


def test_backward_full_training_shape_sampled_heads():
    # B8 H8 T4096 d128 bf16: every head runs on the GPU; heads 0 and 7 of
    # batches 0 and 5 are checked against the oracle
    kla = _kla()
    inp = kla_inputs.make_prefill(kla_inputs.TRAIN.with_(h0_std=0.05), device="cuda")
    do, dh = _grad_inputs(inp, 480)
    got = kla.chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], do, dh, inp["eps"],
                        inp["h0"])
    torch.cuda.synchronize()
    bi = torch.tensor([0, 5], device="cuda")
    hi = torch.tensor([0, 7], device="cuda")
    tok = lambda t: t.index_select(0, bi).index_select(2, hi)
    st = lambda t: t.index_select(0, bi).index_select(1, hi)
    ref = oracle.kla_oracle_backward(*(tok(inp[n]) for n in ("q", "k", "v", "g", "eta")), inp["eps"],
                                     st(inp["h0"]), tok(do), st(dh))
    for n in GRADS:
        e = rel_err(st(got[n]) if n == "dh0" else tok(got[n]), ref[n])
        assert e <= TOL["bf16"], f"{n}: rel err {e:.3e}"
