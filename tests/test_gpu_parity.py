"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element."""
import math

import numpy as np
import pytest
import torch

import kla_inputs
import oracle
from tests.parity_utils import TOL, gpu_prefill, oracle_prefill, rel_err, to_cuda

pytestmark = pytest.mark.gpu


def _check_prefill(inp, io, heads=None, want_hT=True):
    o, hT = gpu_prefill(inp, want_hT=want_hT)
    o_ref, h_ref = oracle_prefill(inp, heads=heads)
    if heads is not None:
        idx = torch.as_tensor(heads, device=o.device)
        o = o.index_select(2, idx)
        hT = hT.index_select(1, idx) if hT is not None else None
    eo = rel_err(o, o_ref)
    assert eo <= TOL[io], f"o rel err {eo:.3e} > {TOL[io]}"
    if want_hT:
        eh = rel_err(hT, h_ref)
        assert eh <= TOL[io], f"hT rel err {eh:.3e} > {TOL[io]}"
    return o, hT


def test_tiny_fp32_case():
    inp = kla_inputs.make_prefill(kla_inputs.TINY, device="cuda")
    _check_prefill(inp, "fp32")


def test_projection_fp32_case():
    inp = kla_inputs.make_prefill(kla_inputs.PROJECTION, device="cuda")
    _check_prefill(inp, "fp32")


def test_projection_constraint_on_gpu():
    """eta=1, eps=0, g=0: every S_t satisfies S_t^T k_t = v_t.  Reading out
    with q := k gives o_t = S_t^T k_t, which must equal v_t for every t."""
    inp = kla_inputs.make_prefill(kla_inputs.PROJECTION, device="cuda")
    inp["q"] = inp["k"].clone()
    o, _ = gpu_prefill(inp, want_hT=False)
    err = rel_err(o, inp["v"].double().cpu().numpy())
    assert err <= TOL["fp32"], err


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130, 257])
def test_ragged_lengths_with_h0(io, T):
    case = kla_inputs.TINY.with_(T=T, B=2, H=3, dk=128, dv=128, io=io, h0_std=0.05, seed=100 + T)
    inp = kla_inputs.make_prefill(case, device="cuda")
    _check_prefill(inp, io)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_head_dims(dk, dv, io):
    case = kla_inputs.TINY.with_(T=200, B=1, H=2, dk=dk, dv=dv, io=io, h0_std=0.02, seed=7)
    inp = kla_inputs.make_prefill(case, device="cuda")
    _check_prefill(inp, io)


def test_projection_gates_bf16_long():
    """bf16 I/O, eps = 0, eta = 1, g = 0 (no decay at all): the hardest case
    for error accumulation through the carry."""
    case = kla_inputs.PROJECTION.with_(io="bf16", T=2048, B=1, H=4, seed=9)
    inp = kla_inputs.make_prefill(case, device="cuda")
    _check_prefill(inp, "bf16")


def test_empty_sequence_copies_h0():
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(T=0, B=2, H=2, h0_std=1.0)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], inp["h0"])
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(hT, inp["h0"])
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(hT) == 0


def test_no_final_state_requested():
    inp = kla_inputs.make_prefill(kla_inputs.TINY.with_(T=100, io="bf16"), device="cuda")
    _check_prefill(inp, "bf16", want_hT=False)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_split_sequence_equals_whole(io):
    """fwd(x[:T1]) -> hT1, then fwd(x[T1:], h0=hT1) reproduces fwd(x)."""
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(T=300, B=2, H=2, dk=128, dv=128, io=io, h0_std=0.1, seed=31)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], inp["h0"])
    T1 = 97
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, h1 = kla.chunk_fwd(*(sl(inp[n], 0, T1) for n in ("q", "k", "v", "g", "eta")), inp["eps"], inp["h0"])
    o2, h2 = kla.chunk_fwd(*(sl(inp[n], T1, 300) for n in ("q", "k", "v", "g", "eta")), inp["eps"], h1)
    torch.cuda.synchronize()
    tol = TOL[io]
    assert rel_err(torch.cat([o1, o2], 1), o.double().cpu().numpy()) <= tol
    assert rel_err(h2, hT.double().cpu().numpy()) <= tol


def test_hT_may_alias_h0():
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(T=130, B=1, H=2, io="fp32", h0_std=0.1, seed=3)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o_ref, h_ref = oracle_prefill(inp)
    S = inp["h0"].clone()
    o = torch.empty_like(inp["v"])
    ws = kla.alloc_workspace(1, 130, 2, 64, 64, io=kla.KLA_IO_FP32)
    kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], S, o, S, ws)
    torch.cuda.synchronize()
    assert rel_err(S, h_ref) <= TOL["fp32"]
    assert rel_err(o, o_ref) <= TOL["fp32"]


def test_workspace_reports_no_device_error():
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(kla_inputs.TINY.with_(io="bf16"), device="cuda")
    ws = kla.alloc_workspace(1, 256, 2, 64, 64)
    o = torch.empty_like(inp["v"])
    kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], None, o, None, ws)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK


# ---------------------------------------------------------------- decode

def _decode_case(io, B=3, H=5, dk=128, dv=128, steps=6, seed=41):
    return kla_inputs.DECODE.with_(B=B, H=H, dk=dk, dv=dv, steps=steps, io=io, seed=seed)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128), (128, 64)])
def test_decode_steps_match_oracle(io, dk, dv):
    import chunked_delta_rule_kla_gb300 as kla
    case = _decode_case(io, dk=dk, dv=dv)
    inp = kla_inputs.make_decode(case, device="cuda")
    S = inp["S"].clone()
    outs = []
    for t in range(case.steps):
        outs.append(kla.decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["g"][t],
                                    inp["eta"][t], S, inp["eps"]))
    torch.cuda.synchronize()
    # the decode loop is the recurrence over the steps: a T=steps oracle run
    tr = lambda x: x.transpose(0, 1).contiguous()
    o_ref, S_ref = oracle.kla_oracle_forward(tr(inp["q"]), tr(inp["k"]), tr(inp["v"]), tr(inp["g"]),
                                             tr(inp["eta"]), inp["eps"], inp["S"])
    o = torch.stack(outs, 1)  # [B,steps,H,dv]
    assert rel_err(o, o_ref) <= TOL[io]
    assert rel_err(S, S_ref) <= TOL[io]


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_prefill_then_decode_equals_longer_prefill(io):
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(T=140, B=2, H=2, dk=128, dv=128, io=io, h0_std=0.05, seed=55)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o_ref, h_ref = oracle_prefill(inp)
    Tp = 131
    sl = lambda n: inp[n][:, :Tp].contiguous()
    o_pre, S = kla.chunk_fwd(sl("q"), sl("k"), sl("v"), sl("g"), sl("eta"), inp["eps"], inp["h0"])
    outs = [o_pre]
    for t in range(Tp, 140):
        pick = lambda n: inp[n][:, t].contiguous()
        outs.append(kla.decode_step(pick("q"), pick("k"), pick("v"), pick("g"), pick("eta"), S,
                                    inp["eps"])[:, None])
    torch.cuda.synchronize()
    assert rel_err(torch.cat(outs, 1), o_ref) <= TOL[io]
    assert rel_err(S, h_ref) <= TOL[io]


def test_decode_empty_batch_is_noop():
    import chunked_delta_rule_kla_gb300 as kla
    z = torch.empty((0, 4, 128), device="cuda", dtype=torch.bfloat16)
    g = torch.empty((0, 4), device="cuda")
    S = torch.empty((0, 4, 128, 128), device="cuda")
    kla.decode_step(z, z, z, g, g, S)


@pytest.mark.parametrize("io,B,H,T,segments", [("bf16", 2, 5, 300, 0), ("bf16", 1, 3, 4096, 4),
                                               ("fp32", 2, 3, 130, 0), ("bf16", 4, 25, 2048, 0)])
def test_permuting_heads_and_batch_permutes_outputs(io, B, H, T, segments):
    """Heads and batch entries are independent: running the call on inputs
    whose (b, h) are permuted gives the outputs permuted the same way, bit
    for bit (each head's work does not depend on where it sits)."""
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(B=B, T=T, H=H, dk=128, dv=128, io=io, h0_std=0.05, seed=400 + H)
    inp = kla_inputs.make_prefill(case, device="cuda")
    gen = torch.Generator().manual_seed(7)
    pb = torch.randperm(B, generator=gen).cuda()
    ph = torch.randperm(H, generator=gen).cuda()

    def perm_tok(x):   # [B, T, H, ...]
        return x.index_select(0, pb).index_select(2, ph).contiguous()

    def perm_state(x):  # [B, H, ...]
        return x.index_select(0, pb).index_select(1, ph).contiguous()

    def run(d):
        o = torch.empty((B, T, H, 128), dtype=d["q"].dtype, device="cuda")
        hT = torch.empty((B, H, 128, 128), device="cuda")
        if segments:
            ws = kla.alloc_workspace(B, T, H, 128, 128, segments=segments)
            kla.kla_chunk_fwd_scan(d["q"], d["k"], d["v"], d["g"], d["eta"], d["eps"], d["h0"], o, hT, ws,
                                   segments)
        else:
            ws = kla.alloc_workspace(B, T, H, 128, 128, io=kla.KLA_IO_BF16 if io == "bf16" else kla.KLA_IO_FP32)
            kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["eta"], d["eps"], d["h0"], o, hT, ws)
        assert kla.kla_workspace_check(ws) == kla.KLA_OK
        return o, hT

    o, hT = run(inp)
    pinp = dict(inp)
    for n in ("q", "k", "v", "g", "eta"):
        pinp[n] = perm_tok(inp[n])
    pinp["h0"] = perm_state(inp["h0"])
    o2, hT2 = run(pinp)
    assert torch.equal(o2, perm_tok(o))
    assert torch.equal(hT2, perm_state(hT))
