"""kla_chunk_fwd_noalloc against kla_chunk_fwd and against the oracle.

Some callers may not allocate device memory: a plugin inside a framework that
owns every device allocation, or a serving loop that fixes its memory budget
at start-up.  kla_chunk_fwd_noalloc serves them with scratch built into the
library instead of a caller-provided workspace.  This test calls it through
the C ABI twice in a row, on different inputs, and checks each result against
kla_chunk_fwd's (the entry point that takes a workspace) and against the fp64
oracle, within the bf16 tolerance of the other parity tests; it also checks
that the call allocates nothing through torch.  A second case fills the
built-in array almost to its 16 MiB limit.  The file sorts last so that a run
stopping at its first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import kla_inputs
from tests.parity_utils import TOL, oracle_prefill, rel_err

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc_call(lib, kla, case, inp, o, hT):
    return lib.kla_chunk_fwd_noalloc(
        _p(inp["q"]), _p(inp["k"]), _p(inp["v"]), _p(inp["g"]), _p(inp["eta"]),
        ctypes.c_float(inp["eps"]), _p(inp["h0"]), _p(o), _p(hT),
        case.B, case.T, case.H, case.dk, case.dv, 64, kla.KLA_IO_BF16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import chunked_delta_rule_kla_gb300 as kla
    lib = kla.load_library()
    for seed in (71, 72):
        case = kla_inputs.TINY.with_(B=2, H=3, T=200, dk=128, dv=128, io="bf16", h0_std=0.05,
                                     seed=seed)
        inp = kla_inputs.make_prefill(case, device="cuda")
        o_or, h_or = oracle_prefill(inp)
        o_ref, h_ref = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"],
                                     inp["eps"], inp["h0"])
        o = torch.full_like(o_ref, float("nan"))
        hT = torch.full_like(h_ref, float("nan"))
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated()
        rc = _noalloc_call(lib, kla, case, inp, o, hT)
        torch.cuda.synchronize()
        assert rc == kla.KLA_OK, kla.kla_status_string(rc)
        assert torch.cuda.memory_allocated() == allocated
        assert lib.kla_chunk_fwd_noalloc_check(None) == kla.KLA_OK   # no device wait ran out
        assert rel_err(o, o_ref.double().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(hT, h_ref.double().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(o, o_or) <= TOL["bf16"]
        assert rel_err(hT, h_or) <= TOL["bf16"]


def test_noalloc_just_under_its_limit():
    """One head whose records nearly fill the 16 MiB array (about 650
    chunks), against the oracle."""
    import chunked_delta_rule_kla_gb300 as kla
    lib = kla.load_library()
    limit = 16 << 20
    T = 64
    while lib.kla_chunk_fwd_workspace_bytes(1, T + 64, 1, 128, 128, 64, kla.KLA_IO_BF16) <= limit:
        T += 64
    T -= 17   # a ragged last chunk
    assert lib.kla_chunk_fwd_workspace_bytes(1, T, 1, 128, 128, 64, kla.KLA_IO_BF16) > limit - 64 * 25344
    case = kla_inputs.TINY.with_(B=1, H=1, T=T, dk=128, dv=128, io="bf16", h0_std=0.05, seed=73)
    inp = kla_inputs.make_prefill(case, device="cuda")
    o = torch.full((1, T, 1, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    hT = torch.full((1, 1, 128, 128), float("nan"), device="cuda")
    rc = _noalloc_call(lib, kla, case, inp, o, hT)
    torch.cuda.synchronize()
    assert rc == kla.KLA_OK, kla.kla_status_string(rc)
    o_or, h_or = oracle_prefill(inp)
    assert rel_err(o, o_or) <= TOL["bf16"]
    assert rel_err(hT, h_or) <= TOL["bf16"]


def test_noalloc_reports_argument_errors():
    import chunked_delta_rule_kla_gb300 as kla
    lib = kla.load_library()
    rc = lib.kla_chunk_fwd_noalloc(None, None, None, None, None, ctypes.c_float(1e-6), None,
                                   None, None, 1, 64, 1, 128, 128, 64, kla.KLA_IO_BF16, None)
    assert rc == kla.KLA_ERR_INVALID_ARG
    rc = lib.kla_chunk_fwd_noalloc(None, None, None, None, None, ctypes.c_float(1e-6), None,
                                   None, None, 1, 64, 1, 96, 128, 64, kla.KLA_IO_BF16, None)
    assert rc == kla.KLA_ERR_UNSUPPORTED
