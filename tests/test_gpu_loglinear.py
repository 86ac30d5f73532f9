"""GPU parity of the Log-Linear gated delta rule (kla_loglinear_fwd) against
the oracle, which writes the buckets out by origin token."""
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


def _inputs(io, B, T, H, dk, dv, seed):
    case = kla_inputs.TINY.with_(B=B, T=T, H=H, dk=dk, dv=dv, io=io, seed=seed)
    inp = kla_inputs.make_prefill(case, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 1)
    L = oracle.loglinear_num_levels(T)
    lam = torch.empty((B, T, H, L), device="cuda").uniform_(0.2, 1.5, generator=gen)
    return inp, lam


def _check(io, B, T, H, dk, dv, seed, direct=False, heads=None, tweak=None):
    kla = _kla()
    inp, lam = _inputs(io, B, T, H, dk, dv, seed)
    if tweak is not None:
        tweak(inp)
    beta = kla.KLA_BETA_DIRECT if direct else kla.KLA_BETA_KACZMARZ
    if direct:
        inp["k"] = torch.nn.functional.normalize(inp["k"].float(), dim=-1).to(inp["k"].dtype)
    io = kla.KLA_IO_BF16 if io == "bf16" else kla.KLA_IO_FP32
    ws = torch.empty(kla.kla_loglinear_workspace_bytes(B, T, H, dk, dv, 64, io), dtype=torch.uint8,
                     device="cuda")
    o = kla.loglinear_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], lam, inp["eps"], beta=beta,
                          workspace=ws)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK      # no device wait ran out
    names = ("q", "k", "v", "g", "eta")
    sel = {n: inp[n] for n in names}
    lam_s = lam
    if heads is not None:
        idx = torch.as_tensor(heads, device="cuda")
        sel = {n: t.index_select(2, idx) for n, t in sel.items()}
        lam_s = lam.index_select(2, idx)
        o = o.index_select(2, idx)
    ref = oracle.kla_oracle_loglinear_forward(*(sel[n] for n in names), lam_s, inp["eps"],
                                              beta_direct=direct)
    e = rel_err(o, ref)
    tol = TOL["bf16" if io == kla.KLA_IO_BF16 else "fp32"]
    assert e <= tol, f"o rel err {e:.3e} > {tol}"


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("T", [1, 5, 64, 65, 130, 200, 520])
def test_loglinear_lengths(io, T):
    _check(io, 1, T, 2, 128, 128, 600 + T)


@pytest.mark.parametrize("dk,dv", [(64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_loglinear_head_dims(io, dk, dv):
    _check(io, 2, 300, 2, dk, dv, 700 + dk + dv)


@pytest.mark.parametrize("io", ["fp32", "bf16"])
def test_loglinear_direct_step_size(io):
    _check(io, 1, 260, 2, 128, 128, 720, direct=True)


def test_loglinear_unit_weights_equal_chunk_fwd():
    # lambda = 1 sums the buckets back into the ordinary state: kla_chunk_fwd's output
    kla = _kla()
    inp, lam = _inputs("fp32", 2, 333, 2, 128, 128, 730)
    lam = torch.ones_like(lam)
    o = kla.loglinear_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], lam, inp["eps"])
    o2, _ = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], None)
    torch.cuda.synchronize()
    assert rel_err(o, o2.double().cpu().numpy()) <= 1e-4


def test_loglinear_batches_and_task_groups():
    # bf16 d128 (the tensor-core path): 21 chunks, so the passes of levels
    # 7..11 run several 16-chunk groups and end in a ragged chunk; B = 2
    _check("bf16", 2, 1300, 3, 128, 128, 760)


def test_loglinear_more_level_tasks_than_sms():
    # B4 H8 T2048: 224 level-pass tasks, more than one per SM, so tasks of all
    # four levels queue behind one another; two heads checked
    _check("bf16", 4, 2048, 8, 128, 128, 780, heads=[0, 5])


def test_loglinear_strong_decay_chunk():
    # chunk 2 decays by about 2 per token (a span far above 80): the level
    # passes take the direct P W branch there and the factorised one elsewhere
    def strong(inp):
        g = inp["g"].clone()
        g[:, 128:192] *= 15.0
        inp["g"] = g.contiguous()
    _check("bf16", 1, 600, 2, 128, 128, 770, tweak=strong)


def test_loglinear_training_shape_sampled_heads():
    # B1 H4 T4096 d128 bf16: 64 chunks, level states up to bit 5; two heads checked
    _check("bf16", 1, 4096, 4, 128, 128, 740, heads=[0, 3])


@pytest.mark.parametrize("io", ["fp32", "bf16"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_loglinear_decode_steps_match_oracle(io, dk, dv):
    # T decode steps from zero states give the Log-Linear outputs of the whole sequence
    kla = _kla()
    B, T, H = 2, 150, 3
    inp, lam = _inputs(io, B, T, H, dk, dv, 750 + dk)
    L = lam.shape[-1]
    states = torch.zeros((B, H, L, dk, dv), device="cuda")
    outs = []
    for t in range(T):
        pick = lambda n: inp[n][:, t].contiguous()
        o = torch.empty((B, H, dv), dtype=inp["q"].dtype, device="cuda")
        kla.kla_loglinear_decode_step(pick("q"), pick("k"), pick("v"), pick("g"), pick("eta"),
                                      lam[:, t].contiguous(), inp["eps"], states, t, o)
        outs.append(o)
    torch.cuda.synchronize()
    ref = oracle.kla_oracle_loglinear_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], lam,
                                              inp["eps"])
    assert rel_err(torch.stack(outs, 1), ref) <= TOL[io]


def test_loglinear_bench_shape_sampled_sequences():
    # B8 H8 T4096, the shape and launch configuration the bench times (960
    # level-pass tasks, 2,048 chunk pairs); two (batch, head) sequences checked
    kla = _kla()
    case = kla_inputs.TRAIN
    inp = kla_inputs.make_prefill(case, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(790)
    L = oracle.loglinear_num_levels(case.T)
    lam = torch.empty((case.B, case.T, case.H, L), device="cuda").uniform_(0.2, 1.5, generator=gen)
    ws = torch.empty(kla.kla_loglinear_workspace_bytes(case.B, case.T, case.H, 128, 128, 64, kla.KLA_IO_BF16),
                     dtype=torch.uint8, device="cuda")
    o = kla.loglinear_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], lam, inp["eps"], workspace=ws)
    assert kla.kla_workspace_check(ws) == kla.KLA_OK
    for b, h in ((0, 0), (7, 5)):
        sl = lambda x: x[b:b + 1, :, h:h + 1]  # noqa: E731
        ref = oracle.kla_oracle_loglinear_forward(*(sl(inp[n]) for n in ("q", "k", "v", "g", "eta")), sl(lam),
                                                  inp["eps"])
        e = rel_err(sl(o), ref)
        assert e <= TOL["bf16"], f"(b={b}, h={h}) rel err {e:.3e}"


def test_loglinear_decode_bench_shape_sampled_heads():
    # B64 H16 d128, tokens 0..1023 from zero states (the bench's decode run);
    # two heads checked against the oracle over the whole sequence
    kla = _kla()
    case = kla_inputs.DECODE
    steps = 1024
    dec = kla_inputs.make_decode(case, device="cuda", steps=steps)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(791)
    L = oracle.loglinear_num_levels(steps)
    lam = torch.empty((steps, case.B, case.H, L), device="cuda").uniform_(0.2, 1.5, generator=gen)
    states = torch.zeros((case.B, case.H, L, 128, 128), device="cuda")
    o = torch.empty((steps, case.B, case.H, 128), dtype=torch.bfloat16, device="cuda")
    for t in range(steps):
        kla.kla_loglinear_decode_step(dec["q"][t], dec["k"][t], dec["v"][t], dec["g"][t], dec["eta"][t], lam[t],
                                      dec["eps"], states, t, o[t])
    torch.cuda.synchronize()
    for b, h in ((0, 0), (63, 15)):
        seq = lambda x: x[:, b:b + 1, h:h + 1].transpose(0, 1).contiguous()  # noqa: E731  [1, T, 1, ...]
        ref = oracle.kla_oracle_loglinear_forward(*(seq(dec[n]) for n in ("q", "k", "v", "g", "eta")), seq(lam),
                                                  dec["eps"])
        e = rel_err(seq(o), ref)
        assert e <= TOL["bf16"], f"(b={b}, h={h}) rel err {e:.3e}"
