"""Parity at the full workload sizes, through the same calls bench.py times.

- training-shape prefill B8 H8 T4096 d128 bf16: every head against the oracle;
- long-context prefill B1 H16 T131072 d128 bf16: sampled heads, o and hT;
- decode B64 H16 d128 bf16, 1024 consecutive steps: sampled heads, every
  step's o and the final state;
- the training shape under the direct step size with unit-norm keys, and
  DeltaKATA on it (p = 15 raw values to 128 features): sampled heads.
"""
import pytest
import torch

import kla_inputs
import oracle
from tests.parity_utils import TOL, oracle_prefill, rel_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _prefill(inp):
    import chunked_delta_rule_kla_gb300 as kla
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], inp["h0"])
    torch.cuda.synchronize()
    return o, hT


def test_train_prefill_full():
    inp = kla_inputs.make_prefill(kla_inputs.TRAIN, device="cuda")
    o, hT = _prefill(inp)
    o_ref, h_ref = oracle_prefill(inp)
    assert rel_err(o, o_ref) <= TOL["bf16"]
    assert rel_err(hT, h_ref) <= TOL["bf16"]


def test_long_prefill_sampled_heads():
    inp = kla_inputs.make_prefill(kla_inputs.LONG, device="cuda")
    o, hT = _prefill(inp)
    heads = [0, 7, 15]
    o_ref, h_ref = oracle_prefill(inp, heads=heads)
    idx = torch.as_tensor(heads, device="cuda")
    assert rel_err(o.index_select(2, idx), o_ref) <= TOL["bf16"]
    assert rel_err(hT.index_select(1, idx), h_ref) <= TOL["bf16"]


def test_decode_1024_steps_sampled_heads():
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.DECODE
    inp = kla_inputs.make_decode(case, device="cuda")
    S = inp["S"].clone()
    n = case.steps
    o_all = torch.empty((n, case.B, case.H, case.dv), dtype=torch.bfloat16, device="cuda")
    for t in range(n):
        kla.kla_decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["g"][t], inp["eta"][t],
                            inp["eps"], S, o_all[t])
    torch.cuda.synchronize()
    pairs = [(0, 0), (5, 3), (17, 15), (32, 8), (63, 15), (63, 0)]
    bs = torch.tensor([p[0] for p in pairs], device="cuda")
    hs = torch.tensor([p[1] for p in pairs], device="cuda")
    pick = lambda x: x[:, bs, hs].transpose(0, 1).unsqueeze(2).contiguous()  # [P, n, 1, d]
    o_ref, S_ref = oracle.kla_oracle_forward(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]),
                                             inp["g"][:, bs, hs].T.unsqueeze(2),
                                             inp["eta"][:, bs, hs].T.unsqueeze(2), inp["eps"],
                                             inp["S"][bs, hs].unsqueeze(1))
    assert rel_err(pick(o_all), o_ref) <= TOL["bf16"]
    assert rel_err(S[bs, hs].unsqueeze(1), S_ref) <= TOL["bf16"]


def test_gdn_train_prefill_sampled_heads():
    # the training shape under the direct step size with unit-norm keys (the bench's GDN line)
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(kla_inputs.GDN_TRAIN, device="cuda")
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], inp["h0"],
                          beta=kla.KLA_BETA_DIRECT)
    torch.cuda.synchronize()
    heads = [1, 6]
    idx = torch.as_tensor(heads, device="cuda")
    sel = {n: inp[n].index_select(2, idx) for n in ("q", "k", "v", "g", "eta")}
    h0 = inp["h0"].index_select(1, idx) if inp["h0"] is not None else None
    o_ref, h_ref = oracle.kla_oracle_forward(sel["q"], sel["k"], sel["v"], sel["g"], sel["eta"], inp["eps"], h0,
                                             beta_direct=True)
    assert rel_err(o.index_select(2, idx), o_ref) <= TOL["bf16"]
    assert rel_err(hT.index_select(1, idx), h_ref) <= TOL["bf16"]


def test_deltakata_train_prefill_sampled_sequences():
    # DeltaKATA at the bench's shape: p = 15 raw values -> 128 PSD features, B8 H8 T4096
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.TRAIN
    inp = kla_inputs.make_prefill(case, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(case.seed + 2000)
    q = torch.randn((case.B, case.T, case.H, 15), generator=gen, device="cuda").mul(0.4).to(torch.bfloat16)
    u = torch.randn((case.B, case.T, case.H, 15), generator=gen, device="cuda")
    k = (u / u.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    o, hT = kla.deltakata(q, k, inp["v"], inp["g"], inp["eta"], inp["eps"])
    torch.cuda.synchronize()
    for b, h in ((0, 2), (6, 7)):
        sl = lambda x: x[b:b + 1, :, h:h + 1]  # noqa: E731
        fq = oracle.kla_oracle_psd_features(sl(q), 128)
        fk = oracle.kla_oracle_psd_features(sl(k), 128)
        o_ref, h_ref = oracle.kla_oracle_forward(fq, fk, sl(inp["v"]), sl(inp["g"]), sl(inp["eta"]), inp["eps"],
                                                 None)
        assert rel_err(sl(o), o_ref) <= TOL["bf16"], (b, h)
        assert rel_err(hT[b:b + 1, h:h + 1], h_ref) <= TOL["bf16"], (b, h)
