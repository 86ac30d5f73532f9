"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding (C ABI) and the fp64 oracle on the same inputs, and measure
max|x - ref| / max|ref|."""
import numpy as np
import torch

import oracle

# Tolerances on max|x - ref| / max|ref| for o and hT: 1e-2 with bf16 I/O,
# 1e-4 with fp32 I/O.
TOL = {"bf16": 1e-2, "fp32": 1e-4}


def rel_err(x, ref) -> float:
    x = x.detach().double().cpu().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    denom = np.abs(ref).max()
    assert np.isfinite(x).all(), "non-finite values in GPU output"
    return float(np.abs(x - ref).max() / denom) if denom > 0 else float(np.abs(x).max())


def oracle_prefill(inp, heads=None, threads=0):
    """Oracle on the exact values the GPU received (optionally a subset of heads)."""
    q, k, v, g, eta, h0 = (inp[n] for n in ("q", "k", "v", "g", "eta", "h0"))
    if heads is not None:
        idx = torch.as_tensor(heads, device=q.device)
        q, k, v = (t.index_select(2, idx) for t in (q, k, v))
        g, eta = (t.index_select(2, idx) for t in (g, eta))
        h0 = h0.index_select(1, idx) if h0 is not None else None
    return oracle.kla_oracle_forward(q, k, v, g, eta, inp["eps"], h0, threads=threads)


def gpu_prefill(inp, want_hT=True, chunk=64):
    import chunked_delta_rule_kla_gb300 as kla
    o, hT = kla.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"],
                          inp["h0"], output_final_state=want_hT, chunk=chunk)
    torch.cuda.synchronize()
    return o, hT


def to_cuda(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
