"""The chunk-level scan (kla_chunk_fwd_scan) against the fp64 oracle.

The scan splits each head's chunks into runs, forms every run's affine state
map [N | M] from [0 | I], combines the runs in order and replays each run
from its true start state.  Its result must match the oracle at every run
count, for every head-dimension pair, with a nonzero h0 and a ragged last
chunk, and agree with the unsegmented path.
"""
import pytest
import torch

import kla_inputs
from tests.parity_utils import TOL, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def _scan(inp, segments):
    import chunked_delta_rule_kla_gb300 as kla
    q, k, v = inp["q"], inp["k"], inp["v"]
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    o = torch.full((B, T, H, dv), float("nan"), dtype=q.dtype, device=q.device)
    hT = torch.full((B, H, dk, dv), float("nan"), dtype=torch.float32, device=q.device)
    ws = kla.alloc_workspace(B, T, H, dk, dv, segments=segments)
    kla.kla_chunk_fwd_scan(q, k, v, inp["g"], inp["eta"], inp["eps"], inp["h0"], o, hT, ws, segments)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK
    return o, hT


@pytest.mark.parametrize("segments", [2, 3, 5, 16, 40])
def test_scan_matches_oracle_ragged_with_h0(segments):
    # 16 chunks, the last one ragged (1000 = 15*64 + 40); 40 runs clamp to 16
    case = kla_inputs.TINY.with_(B=2, H=3, T=1000, dk=128, dv=128, io="bf16", h0_std=0.05, seed=81)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _scan(inp, segments)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_scan_head_dims(dk, dv):
    case = kla_inputs.TINY.with_(B=1, H=2, T=640, dk=dk, dv=dv, io="bf16", h0_std=0.05, seed=82)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _scan(inp, 4)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_scan_agrees_with_unsegmented_path():
    case = kla_inputs.TINY.with_(B=1, H=4, T=4096, dk=128, dv=128, io="bf16", seed=83)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o1, h1 = _scan(inp, 1)
    o8, h8 = _scan(inp, 8)
    ref_o, ref_h = oracle_prefill(inp, heads=[0, 3])
    idx = torch.tensor([0, 3], device="cuda")
    for o, hT in ((o1, h1), (o8, h8)):
        assert rel_err(o.index_select(2, idx), ref_o) <= TOL["bf16"]
        assert rel_err(hT.index_select(1, idx), ref_h) <= TOL["bf16"]
    # both paths round differently but must agree to the same bound
    assert rel_err(o8, o1.double().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(h8, h1.double().cpu().numpy()) <= TOL["bf16"]


def test_scan_long_sequence_few_heads():
    # the regime the scan is for: few heads, many chunks (here 256 chunks, 8 runs)
    case = kla_inputs.LONG.with_(T=16384, H=2, seed=84)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o, hT = _scan(inp, 8)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]
