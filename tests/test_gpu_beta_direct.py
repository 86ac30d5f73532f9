"""GPU parity of the direct step size (KLA_BETA_DIRECT: beta_t = eta_t as given,
the Gated DeltaNet parameterisation the KLA page sets against its Kaczmarz step)
on every prefill path and on decode, against the fp64 oracle run with the same
rule.  Keys have norms in [0.5, 1.2] and eta lies in (0, 1), so beta ||k||^2 < 2
keeps the recurrence contractive while the two rules give different results."""
import pytest
import torch

import kla_inputs
import oracle
from tests.parity_utils import TOL, rel_err

pytestmark = pytest.mark.gpu

KNORM = (0.5, 1.2)


def _kla():
    import chunked_delta_rule_kla_gb300 as kla
    return kla


def _oracle(inp, heads=None, direct=True):
    q, k, v, g, eta, h0 = (inp[n] for n in ("q", "k", "v", "g", "eta", "h0"))
    if heads is not None:
        idx = torch.as_tensor(heads, device=q.device)
        q, k, v, g, eta = (t.index_select(2, idx) for t in (q, k, v, g, eta))
        h0 = h0.index_select(1, idx) if h0 is not None else None
    return oracle.kla_oracle_forward(q, k, v, g, eta, inp["eps"], h0, beta_direct=direct)


def _run(inp, segments=0):
    kla = _kla()
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    io = kla.KLA_IO_BF16 if q.dtype == torch.bfloat16 else kla.KLA_IO_FP32
    o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device=q.device)
    ws = kla.alloc_workspace(B, T, H, dk, dv, io=io, segments=segments)
    kla.kla_chunk_fwd_ex(q, k, v, inp["g"], inp["eta"], inp["eps"], inp["h0"], o, hT, ws,
                         beta=kla.KLA_BETA_DIRECT, segments=segments)
    torch.cuda.synchronize()
    return o, hT


def _check(inp, io, heads=None, segments=0):
    o, hT = _run(inp, segments)
    o_ref, h_ref = _oracle(inp, heads)
    if heads is not None:
        idx = torch.as_tensor(heads, device=o.device)
        o, hT = o.index_select(2, idx), hT.index_select(1, idx)
    eo, eh = rel_err(o, o_ref), rel_err(hT, h_ref)
    assert eo <= TOL[io], f"o rel err {eo:.3e} > {TOL[io]}"
    assert eh <= TOL[io], f"hT rel err {eh:.3e} > {TOL[io]}"
    return o, hT


def _case(io, **kw):
    base = kla_inputs.TINY.with_(B=2, T=257, H=3, dk=128, dv=128, io=io, h0_std=0.05,
                                 knorm=KNORM, seed=901)
    return base.with_(**kw)


@pytest.mark.parametrize("io", ["bf16", "fp32"])
@pytest.mark.parametrize("T", [1, 64, 130, 257])
def test_direct_beta_d128(io, T):
    # bf16: the fused prep + carry grid; fp32: the CUDA-core chunk kernel
    inp = kla_inputs.make_prefill(_case(io, T=T, seed=900 + T), device="cuda")
    _check(inp, io)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
def test_direct_beta_other_head_dims(dk, dv):
    # bf16 with d_k or d_v = 64: a prep grid, then a carry grid
    inp = kla_inputs.make_prefill(_case("bf16", dk=dk, dv=dv, T=200, seed=910 + dk + dv),
                                  device="cuda")
    _check(inp, "bf16")


def test_direct_beta_scan():
    # three runs of the chunk-level scan over a 40-chunk sequence
    inp = kla_inputs.make_prefill(_case("bf16", B=1, H=2, T=64 * 40 - 7, seed=921), device="cuda")
    _check(inp, "bf16", segments=3)


def test_direct_beta_chunk_ranges():
    # 77 heads and 33 chunks: chunk ranges that hand the state over; three heads checked
    inp = kla_inputs.make_prefill(_case("bf16", B=1, H=77, T=64 * 32 + 5, h0_std=0.0, seed=922),
                                  device="cuda")
    _check(inp, "bf16", heads=[0, 38, 76])


def test_deltanet_without_decay():
    # DeltaNet: the direct step size with no decay (g = 0)
    inp = kla_inputs.make_prefill(_case("bf16", T=190, seed=923), device="cuda")
    inp["g"] = torch.zeros_like(inp["g"])
    _check(inp, "bf16")


def test_direct_differs_from_kaczmarz():
    # with key norms away from 1 the two step-size rules must give different outputs
    kla = _kla()
    inp = kla_inputs.make_prefill(_case("bf16", T=130, seed=924), device="cuda")
    o_direct, _ = _run(inp)
    o_kacz, _ = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"],
                              inp["h0"])
    torch.cuda.synchronize()
    o_ref_kacz, _ = _oracle(inp, direct=False)
    assert rel_err(o_kacz, o_ref_kacz) <= TOL["bf16"]
    assert rel_err(o_direct, o_ref_kacz) > 10 * TOL["bf16"]


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_direct_beta_decode(io, dk, dv):
    kla = _kla()
    case = kla_inputs.DECODE.with_(B=3, H=5, dk=dk, dv=dv, steps=6, io=io, knorm=KNORM, seed=931)
    inp = kla_inputs.make_decode(case, device="cuda")
    S = inp["S"].clone()
    outs = [kla.decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["g"][t], inp["eta"][t], S,
                            inp["eps"], beta=kla.KLA_BETA_DIRECT) for t in range(case.steps)]
    torch.cuda.synchronize()
    tr = lambda x: x.transpose(0, 1).contiguous()
    o_ref, S_ref = oracle.kla_oracle_forward(tr(inp["q"]), tr(inp["k"]), tr(inp["v"]), tr(inp["g"]),
                                             tr(inp["eta"]), inp["eps"], inp["S"], beta_direct=True)
    assert rel_err(torch.stack(outs, 1), o_ref) <= TOL[io]
    assert rel_err(S, S_ref) <= TOL[io]


def test_direct_prefill_then_decode():
    kla = _kla()
    inp = kla_inputs.make_prefill(_case("bf16", T=140, seed=932), device="cuda")
    o_ref, h_ref = _oracle(inp)
    Tp = 131
    sl = lambda n: inp[n][:, :Tp].contiguous()
    o_pre, S = kla.chunk_fwd(sl("q"), sl("k"), sl("v"), sl("g"), sl("eta"), inp["eps"], inp["h0"],
                             beta=kla.KLA_BETA_DIRECT)
    outs = [o_pre]
    for t in range(Tp, 140):
        pick = lambda n: inp[n][:, t].contiguous()
        outs.append(kla.decode_step(pick("q"), pick("k"), pick("v"), pick("g"), pick("eta"), S,
                                    inp["eps"], beta=kla.KLA_BETA_DIRECT)[:, None])
    torch.cuda.synchronize()
    assert rel_err(torch.cat(outs, 1), o_ref) <= TOL["bf16"]
    assert rel_err(S, h_ref) <= TOL["bf16"]
