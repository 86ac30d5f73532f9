"""Paths the configurations do not reach on their own.

- Strong decay: with g about -2 per token a chunk's decay span
  gam_0 - gam_63 exceeds 80, so every kernel takes its unfactorised branch
  (one exponential per decay factor) instead of exp(gam_r - gam_m) *
  exp(gam_m - gam_s).
- One fused grid: d_k = d_v = 128 without a scan and with at most 76 heads
  runs prep lanes and carries in one cooperative grid, the carries waiting
  on per-chunk ready flags; here with a nonzero h0, with and without hT,
  with 76 heads (the most the grid takes) and with a single head.
- Chunk ranges: with 77 to 136 heads and >= 32 chunks the carry runs in
  growing chunk ranges, the state passing between ranges through the
  workspace; here with a nonzero h0 and without hT (the handoff buffer)
  and with hT.
"""
import pytest
import torch

import kla_inputs
from tests.parity_utils import TOL, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def _run(inp, segments=0, want_hT=True):
    import chunked_delta_rule_kla_gb300 as kla
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = torch.full((B, T, H, dv), float("nan"), dtype=q.dtype, device=q.device)
    hT = torch.full((B, H, dk, dv), float("nan"), device=q.device) if want_hT else None
    ws = kla.alloc_workspace(B, T, H, dk, dv, segments=segments)
    kla.kla_chunk_fwd_scan(q, k, v, inp["g"], inp["eta"], inp["eps"], inp["h0"], o, hT, ws, segments)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK
    return o, hT


def _strong(inp):
    inp = dict(inp)
    inp["g"] = (inp["g"] * 15.0).contiguous()   # about -2 per token
    span = -inp["g"][:, :64].sum(1).max().item()
    assert span > 80.0, span
    return inp


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64), (64, 128)])
def test_strong_decay(dk, dv):
    case = kla_inputs.TINY.with_(B=1, H=2, T=300, dk=dk, dv=dv, io="bf16", h0_std=0.05, seed=91)
    inp = _strong(kla_inputs.make_prefill(case, device="cuda"))
    o, hT = _run(inp, segments=1)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_strong_decay_through_the_scan():
    case = kla_inputs.TINY.with_(B=1, H=2, T=640, dk=128, dv=128, io="bf16", h0_std=0.05, seed=92)
    inp = _strong(kla_inputs.make_prefill(case, device="cuda"))
    o, hT = _run(inp, segments=3)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


@pytest.mark.parametrize("want_hT", [False, True])
def test_fused_grid_with_h0(want_hT):
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TINY.with_(B=1, H=3, T=64 * 40 - 17, dk=128, dv=128, io="bf16", h0_std=0.05, seed=93)
    assert kla.kla_chunk_fwd_auto_segments(case.B, case.T, case.H, 128, 128) == 1  # no scan
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _run(inp, want_hT=want_hT)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    if want_hT:
        assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_fused_grid_strong_decay():
    case = kla_inputs.TINY.with_(B=2, H=2, T=64 * 36, dk=128, dv=128, io="bf16", h0_std=0.05, seed=94)
    inp = _strong(kla_inputs.make_prefill(case, device="cuda"))
    o, hT = _run(inp)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_fused_grid_most_heads():
    # 76 carries and 76 prep CTAs; a ragged last chunk
    case = kla_inputs.TINY.with_(B=4, H=19, T=64 * 9 - 5, dk=128, dv=128, io="bf16", h0_std=0.05, seed=95)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _run(inp)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


@pytest.mark.parametrize("want_hT", [False, True])
def test_chunk_ranges_with_h0(want_hT):
    import chunked_delta_rule_kla_gb300 as kla
    # 80 heads: too many for the fused grid, few enough for chunk ranges
    case = kla_inputs.TINY.with_(B=2, H=40, T=64 * 33 - 9, dk=128, dv=128, io="bf16", h0_std=0.05, seed=96)
    assert kla.kla_chunk_fwd_auto_segments(case.B, case.T, case.H, 128, 128) == 1  # no scan
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _run(inp, want_hT=want_hT)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    if want_hT:
        assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_fused_grid_single_head():
    # one carry CTA beside 151 prep CTAs, most of whose lanes get no item
    case = kla_inputs.TINY.with_(B=1, H=1, T=64 * 5 + 7, dk=128, dv=128, io="bf16", h0_std=0.05, seed=97)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _run(inp)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]
