"""Bounded device waits: a wait that runs out is reported, the kernel exits
cleanly, and the GPU stays usable.

Every cross-CTA wait of the fused prefill grid (a carry polling the ready flag
of a chunk record that a prep lane publishes) gives up after a limit, records
the error in the workspace's device error record, stops issuing, waits for
its own copies and MMAs and returns; kla_workspace_check then reports
KLA_ERR_DEVICE_TIMEOUT.  To drive that path without faulting anything, the
test builds a variant of the library (in a folder of its own) in which the
prep lanes never publish the flag of one chunk of head 0 -- a flag that
nothing sets -- and the flag wait is cut to 2 ms.  The variant runs in a
child process: the call must come back with KLA_ERR_DEVICE_TIMEOUT at that
chunk, the other heads must still match the oracle, and further calls in the
same process must work.

The decode step's own error record (kla_decode_step_checked) is checked on
the success path against kla_decode_step.
"""
import json
import os
import subprocess
import sys

import pytest
import torch

import kla_inputs
from tests.parity_utils import TOL, rel_err

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
UNPUBLISHED = 3
WHERE_FLAG = 18          # the error-record site of the ready-flag wait

CHILD = r"""
import json, sys
import torch
import chunked_delta_rule_kla_gb300 as kla
import kla_inputs
from tests.parity_utils import oracle_prefill, rel_err

kla.load_library(sys.argv[1])
case = kla_inputs.TINY.with_(B=1, H=4, T=512, dk=128, dv=128, io="bf16", seed=5)
inp = kla_inputs.make_prefill(case, device="cuda")
ws = kla.alloc_workspace(1, 512, 4, 128, 128)
o = torch.zeros((1, 512, 4, 128), dtype=torch.bfloat16, device="cuda")
hT = torch.zeros((1, 4, 128, 128), device="cuda")
kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], None, o, hT, ws)
status = kla.kla_workspace_check(ws)
record = ws[:16].view(torch.int32).cpu().tolist()
o_ref, h_ref = oracle_prefill(inp, heads=[1, 2, 3])
other_heads = max(rel_err(o[:, :, 1:], o_ref), rel_err(hT[:, 1:], h_ref))
# the context is still usable: the same call again, and a synchronize
kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], None, o, hT, ws)
again = kla.kla_workspace_check(ws)
torch.cuda.synchronize()
print(json.dumps(dict(status=status, record=record[:4], other_heads=other_heads, again=again)))
"""


def test_flag_wait_runs_out_and_is_reported():
    import chunked_delta_rule_kla_gb300 as kla
    from chunked_delta_rule_kla_gb300 import _build
    variant = _build.build(
        extra_flags=["-DKLA_TEST_FLAG_WAIT_NS=2000000ull", f"-DKLA_TEST_UNPUBLISHED_CHUNK={UNPUBLISHED}"],
        build_dir=os.path.join(_build.BUILD_DIR, "wait_test"))
    r = subprocess.run([sys.executable, "-c", CHILD, variant], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == kla.KLA_ERR_DEVICE_TIMEOUT
    code, where, block, detail = res["record"]
    assert code == 1 and where == WHERE_FLAG and detail == UNPUBLISHED
    assert res["other_heads"] <= TOL["bf16"]
    assert res["again"] == kla.KLA_ERR_DEVICE_TIMEOUT     # the variant never publishes that flag


CHILD_DELTAKATA = r"""
import json, sys
import torch
import chunked_delta_rule_kla_gb300 as kla
import oracle
from tests.parity_utils import rel_err

kla.load_library(sys.argv[1])
B, T, H, p = 1, 512, 4, 15
gen = torch.Generator(device="cuda")
gen.manual_seed(6)
xq = (torch.randn((B, T, H, p), generator=gen, device="cuda") * 0.4).to(torch.bfloat16)
u = torch.randn((B, T, H, p), generator=gen, device="cuda")
xk = (u / u.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
v = torch.randn((B, T, H, 128), generator=gen, device="cuda").to(torch.bfloat16)
g = torch.nn.functional.logsigmoid(torch.randn((B, T, H), generator=gen, device="cuda") + 2.0)
eta = torch.sigmoid(torch.randn((B, T, H), generator=gen, device="cuda"))
ws = torch.empty(kla.kla_deltakata_fwd_workspace_bytes(B, T, H, p, 128), dtype=torch.uint8, device="cuda")
o = torch.zeros((B, T, H, 128), dtype=torch.bfloat16, device="cuda")
hT = torch.zeros((B, H, 128, 128), device="cuda")
kla.kla_deltakata_fwd(xq, xk, v, g, eta, 1e-6, None, o, hT, ws)
status = kla.kla_workspace_check(ws)
record = ws[:16].view(torch.int32).cpu().tolist()
hs = slice(1, 4)
fq = oracle.kla_oracle_psd_features(xq[:, :, hs], 128)
fk = oracle.kla_oracle_psd_features(xk[:, :, hs], 128)
o_ref, h_ref = oracle.kla_oracle_forward(fq, fk, v[:, :, hs], g[:, :, hs], eta[:, :, hs], 1e-6)
other_heads = max(rel_err(o[:, :, hs], o_ref), rel_err(hT[:, hs], h_ref))
torch.cuda.synchronize()
print(json.dumps(dict(status=status, record=record[:4], other_heads=other_heads)))
"""


def test_flag_wait_runs_out_with_deltakata_inputs():
    # the same bounded flag wait on the feature path (kla_deltakata_fwd)
    import chunked_delta_rule_kla_gb300 as kla
    from chunked_delta_rule_kla_gb300 import _build
    variant = _build.build(
        extra_flags=["-DKLA_TEST_FLAG_WAIT_NS=2000000ull", f"-DKLA_TEST_UNPUBLISHED_CHUNK={UNPUBLISHED}"],
        build_dir=os.path.join(_build.BUILD_DIR, "wait_test"))
    r = subprocess.run([sys.executable, "-c", CHILD_DELTAKATA, variant], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["status"] == kla.KLA_ERR_DEVICE_TIMEOUT
    code, where, block, detail = res["record"]
    assert code == 1 and where == WHERE_FLAG and detail == UNPUBLISHED
    assert res["other_heads"] <= TOL["bf16"]


def test_decode_step_checked_matches_and_reports_no_error():
    import chunked_delta_rule_kla_gb300 as kla
    case = kla_inputs.DECODE.with_(B=3, H=5, dk=128, dv=128, steps=4, io="bf16", seed=17)
    inp = kla_inputs.make_decode(case, device="cuda")
    S1 = inp["S"].clone()
    S2 = inp["S"].clone()
    o1 = torch.empty((3, 5, 128), dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    status = torch.zeros(64, dtype=torch.int32, device="cuda")
    for t in range(case.steps):
        args = (inp["q"][t], inp["k"][t], inp["v"][t], inp["g"][t], inp["eta"][t], inp["eps"])
        kla.kla_decode_step(*args, S1, o1)
        kla.kla_decode_step(*args, S2, o2, status=status)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
    assert torch.equal(S1, S2)
    assert kla.kla_workspace_check(status) == kla.KLA_OK
    assert rel_err(S2, S1.double().cpu().numpy()) == 0.0
