"""Seeded synthetic inputs for the KLA prefill and decode workloads.

This module only draws random numbers with the value distributions of the
workloads.  It holds none of the recurrence's arithmetic, so the CUDA path and
the fp64 oracle can both take their inputs from it.

Recipes (draw order inside one generator: q, k direction, k norm, v, g
pre-activation, eta pre-activation, h0 / S):

  q ~ N(0, 1);  v ~ N(0, 1)
  k = u / ||u|| * r,  u ~ N(0, 1)/sqrt(dk),  ln r ~ U(ln lo, ln hi)
  g = logsigmoid(N(2, 1))   (log-decay, always <= 0)
  eta = sigmoid(N(0, 1))
  h0 ~ N(0, std^2) or zero

"projection" gates set eta = 1, g = 0 (used with eps = 0).

Large cases are drawn on the device with a seeded torch generator, small
ones on the host; the consumer casts q/k/v to the I/O dtype and the oracle
reads the cast values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class PrefillCase:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    io: str              # "bf16" or "fp32" (q, k, v, o); g, eta, h0, hT are fp32
    eps: float
    seed: int
    knorm: tuple = (0.25, 4.0)
    gates: str = "random"  # "random" or "projection"
    h0_std: float = 0.0    # 0 -> h0 absent (zero state)
    chunk: int = 64

    def with_(self, **kw) -> "PrefillCase":
        return replace(self, **kw)


@dataclass(frozen=True)
class DecodeCase:
    name: str
    B: int
    H: int
    dk: int
    dv: int
    steps: int
    io: str
    eps: float
    seed: int
    S_std: float = 0.05
    knorm: tuple = (0.25, 4.0)

    def with_(self, **kw) -> "DecodeCase":
        return replace(self, **kw)


# The five workloads: a tiny fp32 case, the fp32 projection-invariant case,
# the training-shape prefill, the long-context prefill and the decode loop.
TINY = PrefillCase("tiny_fp32_B1H2T256d64", B=1, T=256, H=2, dk=64, dv=64,
                   io="fp32", eps=1e-6, seed=0)
PROJECTION = PrefillCase("projection_fp32_B2H4T1024d128", B=2, T=1024, H=4,
                         dk=128, dv=128, io="fp32", eps=0.0, seed=1,
                         knorm=(0.1, 10.0), gates="projection", h0_std=0.01)
TRAIN = PrefillCase("train_prefill_bf16_B8H8T4096d128", B=8, T=4096, H=8,
                    dk=128, dv=128, io="bf16", eps=1e-6, seed=2)
LONG = PrefillCase("long_prefill_bf16_B1H16T131072d128", B=1, T=131072, H=16,
                   dk=128, dv=128, io="bf16", eps=1e-6, seed=3)
# The training shape under the direct step size (Gated DeltaNet's rule): unit-norm
# keys, as that rule is used with L2-normalised keys, so that eta in (0, 1) keeps
# every step contractive.
GDN_TRAIN = TRAIN.with_(name="gdn_train_prefill_bf16_B8H8T4096d128_unitkeys", knorm=(1.0, 1.0),
                        seed=5)
DECODE = DecodeCase("decode_bf16_B64H16d128_x1024", B=64, H=16, dk=128, dv=128,
                    steps=1024, io="bf16", eps=1e-6, seed=4)

PREFILL_CASES = {0: TINY, 1: PROJECTION, 2: TRAIN, 3: LONG}


def io_torch_dtype(io: str) -> torch.dtype:
    if io == "bf16":
        return torch.bfloat16
    if io == "fp32":
        return torch.float32
    raise ValueError(f"unknown io dtype {io!r}")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _keys(shape, dk, knorm, gen, device):
    u = torch.randn(shape, generator=gen, device=device) / math.sqrt(dk)
    u = u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    lo, hi = knorm
    r = torch.exp(torch.rand(shape[:-1] + (1,), generator=gen, device=device)
                  * (math.log(hi) - math.log(lo)) + math.log(lo))
    return u * r


def _gates(shape, mode, gen, device):
    if mode == "projection":
        return (torch.zeros(shape, device=device), torch.ones(shape, device=device))
    g = F.logsigmoid(torch.randn(shape, generator=gen, device=device) + 2.0)
    eta = torch.sigmoid(torch.randn(shape, generator=gen, device=device))
    return g, eta


def make_prefill(case: PrefillCase, device="cpu") -> dict:
    """Inputs of one prefill call.

    Returns q, k [B,T,H,dk] and v [B,T,H,dv] in the I/O dtype, g and eta
    [B,T,H] fp32, h0 [B,H,dk,dv] fp32 or None, and eps.
    """
    device = torch.device(device)
    gen = _gen(case.seed, device)
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    dt = io_torch_dtype(case.io)
    q = torch.randn((B, T, H, dk), generator=gen, device=device).to(dt)
    k = _keys((B, T, H, dk), dk, case.knorm, gen, device).to(dt)
    v = torch.randn((B, T, H, dv), generator=gen, device=device).to(dt)
    g, eta = _gates((B, T, H), case.gates, gen, device)
    h0 = None
    if case.h0_std > 0:
        h0 = torch.randn((B, H, dk, dv), generator=gen, device=device) * case.h0_std
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(),
                g=g.contiguous(), eta=eta.contiguous(), h0=h0, eps=case.eps)


def make_decode(case: DecodeCase, device="cpu", steps: Optional[int] = None) -> dict:
    """Inputs of ``steps`` consecutive decode calls.

    Returns q, k [steps,B,H,dk] and v [steps,B,H,dv] in the I/O dtype, g and
    eta [steps,B,H] fp32, the initial state S [B,H,dk,dv] fp32, and eps.
    """
    device = torch.device(device)
    n = case.steps if steps is None else int(steps)
    gen = _gen(case.seed, device)
    B, H, dk, dv = case.B, case.H, case.dk, case.dv
    dt = io_torch_dtype(case.io)
    q = torch.randn((n, B, H, dk), generator=gen, device=device).to(dt)
    k = _keys((n, B, H, dk), dk, case.knorm, gen, device).to(dt)
    v = torch.randn((n, B, H, dv), generator=gen, device=device).to(dt)
    g, eta = _gates((n, B, H), "random", gen, device)
    S = torch.randn((B, H, dk, dv), generator=gen, device=device) * case.S_std
    return dict(q=q.contiguous(), k=k.contiguous(), v=v.contiguous(),
                g=g.contiguous(), eta=eta.contiguous(), S=S.contiguous(), eps=case.eps)


__all__ = ["PrefillCase", "DecodeCase", "TINY", "PROJECTION", "TRAIN", "LONG",
           "GDN_TRAIN", "DECODE", "PREFILL_CASES", "make_prefill", "make_decode", "io_torch_dtype"]
