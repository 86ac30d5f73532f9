#!/usr/bin/env python3
"""Throughput of the KLA hot path on one GB300 (or N independent replicas).

Headline workload: the training-shape prefill (B=8, H=8, T=4096,
d_k=d_v=128, bf16 q/k/v/o, fp32 gates, chunk 64) through kla_chunk_fwd:
one step = one call over that batch.  The long-context prefill
(B=1, H=16, T=131072) and the decode loop (B=64, H=16, d=128, fp32 state,
kla_decode_step) are timed in the same run and reported under "secondary", with
the training shape under Gated DeltaNet's step-size rule (kla_chunk_fwd_ex with
KLA_BETA_DIRECT, unit-norm keys), the backward (kla_chunk_bwd) of the
training shape, DeltaKATA (PSD features of 15-value q and k, then
kla_chunk_fwd) and the Log-Linear gated delta rule (kla_loglinear_fwd), both
on the training shape, and Log-Linear decoding (kla_loglinear_decode_step,
1024 tokens of the decode workload's heads).

Timing: W untimed warm-up steps, then exactly K timed steps, each between
CUDA events on the launching stream; L2 is flushed (a 512 MiB write) between
timed steps, outside the events; barrier + synchronize on both sides; max
over ranks.  SM clocks are sampled with nvidia-smi during the run.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only).

Prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kla_inputs  # noqa: E402

METRIC = "prefill tokens/s & % roofline at T=4K/131K; decode tokens/s & HBM GB/s"
FLUSH_BYTES = 512 << 20


# --------------------------------------------------------------- work model

def prefill_work(case):
    """Algorithmic bytes and flops of one prefill call (per launch)."""
    C, dk, dv = case.chunk, case.dk, case.dv
    esz = 2 if case.io == "bf16" else 4
    th = case.B * case.T * case.H
    per_tok_bytes = esz * (2 * dk + 2 * dv) + 8          # q, k, v, o + g, eta
    state_bytes = case.B * case.H * dk * dv * 4          # hT written (h0 absent)
    if case.h0_std > 0:
        state_bytes *= 2
    flops_tok = 4 * C * dk + 2 * C * (dk + dv) + 2 * C * dv + 6 * dk * dv
    return dict(bytes=th * per_tok_bytes + state_bytes, flops=th * flops_tok,
                token_heads=th, tokens=case.B * case.T,
                per_token_head_bytes=per_tok_bytes, per_token_head_flops=flops_tok)


def backward_work(case):
    """Algorithmic bytes of one kla_chunk_bwd call: q, k, v, dO, g, eta read and
    dq, dk, dv, dg, deta written once per token-head; dhT read and dh0 written
    (h0 read too when present) once per head."""
    esz = 2 if case.io == "bf16" else 4
    C, dk, dv = case.chunk, case.dk, case.dv
    th = case.B * case.T * case.H
    per_tok_bytes = esz * (4 * dk + 3 * dv) + 16
    state_bytes = case.B * case.H * dk * dv * 4 * (3 if case.h0_std > 0 else 2)
    # products per token-head: prep 2C(3dk + 2dv), the two carries 10 dk dv,
    # the gradients 2(6C dk + 4C dv + 4 dk dv)
    flops_tok = 2 * C * (9 * dk + 6 * dv) + 18 * dk * dv
    return dict(bytes=th * per_tok_bytes + state_bytes, flops=th * flops_tok, token_heads=th,
                tokens=case.B * case.T, per_token_head_bytes=per_tok_bytes,
                per_token_head_flops=flops_tok)


def decode_work(case):
    heads = case.B * case.H
    esz = 2 if case.io == "bf16" else 4
    per_head = 2 * case.dk * case.dv * 4 + esz * (2 * case.dk + 2 * case.dv) + 8
    return dict(bytes=heads * per_head, flops=heads * (6 * case.dk * case.dv + 4 * case.dk),
                tokens=case.B, per_head_bytes=per_head)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# DRAM bytes (read + write) per call, from one ncu capture of the same
# command (profiles/): every launch of one call, serialised with cold caches,
# so writes still in L2 when a launch ends are not counted.  Refresh these
# whenever the kernels change.
TRAFFIC_BYTES = {
    "train_prefill_bf16_B8H8T4096d128": 453.4e6,
    "gdn_train_prefill_bf16_B8H8T4096d128_unitkeys": 453.2e6,
    "long_prefill_bf16_B1H16T131072d128": 6223.5e6,
    "decode_bf16_B64H16d128_x1024": 73.9e6,
    "loglinear_train_prefill_bf16_B8H8T4096d128": 1760.5e6,
    "bwd_train_prefill_bf16_B8H8T4096d128": 2772.8e6,
    "deltakata_train_prefill_bf16_B8H8T4096d128": 413.7e6,
}


def roofline(work, seconds, peaks, traffic=None):
    t_mem = work["bytes"] / (peaks["hbm"] * 1e9)
    t_flop = work["flops"] / (peaks["bf16"] * 1e12)
    if t_mem >= t_flop:
        ach = work["bytes"] / seconds / 1e9
        return dict(bound="hbm", achieved=round(ach, 1), peak=peaks["hbm"], unit="GB/s",
                    frac=round(ach / peaks["hbm"], 4), traffic=traffic,
                    peak_source=peaks["source"], peak_kind="burst copy bandwidth",
                    roofline_us=round(t_mem * 1e6, 2))
    ach = work["flops"] / seconds / 1e12
    return dict(bound="tensor", achieved=round(ach, 2), peak=peaks["bf16"], unit="TFLOP/s",
                frac=round(ach / peaks["bf16"], 4), traffic=traffic,
                peak_source=peaks["source"], peak_kind="burst bf16 GEMM",
                roofline_us=round(t_flop * 1e6, 2))


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.out = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", "200"]

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(self.cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        reasons = set()
        for r in rows:
            for name, val in zip(self.NAMES, r[5:9]):
                if "Active" in val and "Not" not in val:
                    reasons.add(name)
        loaded = [s for s, p in zip(sm, pw) if pw and p >= 0.5 * max(pw)] or sm
        return dict(sm_mhz=statistics.median(loaded) if loaded else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=sorted(reasons),
                    samples=len(rows), power_w_max=max(pw) if pw else None)


# ------------------------------------------------------------------- timing

def timed_steps(step, K, W, flush_buf, stream):
    """W warm-up steps, then K steps each bracketed by events on `stream`."""
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    for a, b in evs:
        if flush_buf is not None:
            flush_buf.add_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]  # ms


def _dist_on() -> bool:
    return torch.distributed.is_available() and torch.distributed.is_initialized()


def barrier():
    if _dist_on():
        torch.distributed.barrier()


def world_size() -> int:
    return torch.distributed.get_world_size() if _dist_on() else 1


def max_over_ranks(x: float) -> float:
    """Largest x over the ranks (x itself without a process group).  NCCL
    reduces a device tensor, gloo a host tensor."""
    if _dist_on():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def job_throughput(units_per_rank: float, local_seconds: float) -> tuple[float, float]:
    """Whole-job rate for replicas that each process `units_per_rank` units:
    the units of all ranks divided by the slowest rank's time.  Returns
    (units/s over the job, that slowest time in seconds)."""
    slowest = max_over_ranks(local_seconds)
    return units_per_rank * world_size() / slowest, slowest


# ------------------------------------------------------------- native arm

# Kernels of ours launched per ABI call.  kla_chunk_fwd, by dispatch:
#  - chunk-level scan (few heads, long sequences): chunk_prep_kernel, the
#    summary pass, the combine and the carry: 4;
#  - d_k = d_v = 128 with >= 32 chunks and free SMs: chunk ranges, each a
#    prep and a carry launch (the prep of range r+1 overlaps the carry of
#    range r): 2 per range;
#  - otherwise chunk_prep_kernel and the carry: 2;
# plus a 256-byte cudaMemsetAsync of the error record (not a kernel of
# ours).  kla_decode_step launches one kernel.
LAUNCHES_PER_DECODE = 1
MAX_RANGES, RANGE_MIN_CHUNKS, GB300_SMS = 8, 32, 152


def chunk_ranges(nchunks: int) -> int:
    """Number of chunk ranges the library uses (first nchunks/8, at least 4
    chunks, then about 1.25x each; at most MAX_RANGES)."""
    n, lo, size = 0, 0, max(nchunks // 8, 4)
    while lo < nchunks and n < MAX_RANGES:
        lo = nchunks if (n == MAX_RANGES - 1 or lo + size >= nchunks) else lo + size
        n += 1
        size = (size * 5 + 3) // 4
    return n


def prefill_launches(kla, case) -> int:
    segs = kla.kla_chunk_fwd_auto_segments(case.B, case.T, case.H, case.dk, case.dv, case.chunk)
    if segs > 1:
        return 4
    nchunks = -(-case.T // case.chunk)
    if case.dk == 128 and case.dv == 128 and 2 * case.B * case.H <= GB300_SMS:
        return 1   # prep and carry in one cooperative grid
    if (case.dk == 128 and case.dv == 128 and nchunks >= RANGE_MIN_CHUNKS
            and case.B * case.H + 16 <= GB300_SMS):
        return 2 * chunk_ranges(nchunks)
    return 2


def bench_prefill(case, K, W, flush, peaks, stream, e2e=True, direct=False):
    """Time kla_chunk_fwd on ``case`` (kla_chunk_fwd_ex with KLA_BETA_DIRECT when
    ``direct``: the same call under Gated DeltaNet's step-size rule)."""
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(case, device="cuda")
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    o = torch.empty((B, T, H, dv), dtype=inp["q"].dtype, device="cuda")
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    ws = kla.alloc_workspace(B, T, H, dk, dv, case.chunk, kla.KLA_IO_BF16 if case.io == "bf16" else kla.KLA_IO_FP32)

    def step():
        if direct:
            kla.kla_chunk_fwd_ex(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"],
                                 inp["h0"], o, hT, ws, beta=kla.KLA_BETA_DIRECT, chunk=case.chunk,
                                 stream=stream)
        else:
            kla.kla_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"],
                              inp["h0"], o, hT, ws, case.chunk, stream)

    barrier()
    ms = timed_steps(step, K, W, flush, stream)
    barrier()
    assert kla.kla_workspace_check(ws, stream) == kla.KLA_OK
    work = prefill_work(case)
    job_tps, slowest_s = job_throughput(work["tokens"], sum(ms) / len(ms) * 1e-3)
    mean_ms = slowest_s * 1e3
    res = dict(ms_per_step=mean_ms, tokens_per_s=work["tokens"] / (mean_ms * 1e-3),
               job_tokens_per_s=job_tps,
               tflops=work["flops"] / (mean_ms * 1e-3) / 1e12,
               gbps=work["bytes"] / (mean_ms * 1e-3) / 1e9,
               roofline=dict(roofline(work, mean_ms * 1e-3, peaks, TRAFFIC_BYTES.get(case.name)),
                             scope="one kla_chunk_fwd call: all its launches (one fused prep-and-carry grid, or the prep, carry and combine kernels)"), work=work,
               launches=K * prefill_launches(kla, case), min_ms=min(ms),
               segments=kla.kla_chunk_fwd_auto_segments(B, T, H, dk, dv, case.chunk))

    if not e2e:
        del inp, o, hT
        return res
    # end to end through the public API: pinned host inputs -> device -> call
    # -> host, every step.  Steps are pipelined over two device buffer sets:
    # the inputs of step i+1 go up on one copy stream and the outputs of step
    # i-1 come down on another while step i computes (one cudaMemcpyAsync per
    # tensor, ordered by events).
    res["e2e"] = e2e_prefill(kla, case, inp, ws, work, K, stream)
    del inp, o, hT
    return res


def e2e_prefill(kla, case, inp, ws, work, K, stream, sets=2, up_streams=3):
    names = ("q", "k", "v", "g", "eta")
    host = {n: inp[n].cpu().pin_memory() for n in names}
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    dev = [{n: torch.empty_like(inp[n]) for n in names} for _ in range(sets)]
    outs = [(torch.empty((B, T, H, dv), dtype=inp["q"].dtype, device="cuda"),
             torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")) for _ in range(sets)]
    outs_h = [(torch.empty(o.shape, dtype=o.dtype).pin_memory(),
               torch.empty(h.shape, dtype=h.dtype).pin_memory()) for o, h in outs]
    # the large inputs go up on separate copy streams, so that their copies
    # can run on different copy engines at once
    ups = [torch.cuda.Stream() for _ in range(up_streams)]
    up_of = {"q": 0, "k": 1 % up_streams, "v": 2 % up_streams, "g": 0, "eta": 1 % up_streams}
    down = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    loaded = [[ev() for _ in ups] for _ in range(sets)]   # inputs of set j on the device
    consumed = [ev() for _ in range(sets)]    # the call has read set j's inputs and written its outputs
    fetched = [ev() for _ in range(sets)]     # set j's outputs are back on the host
    started = [False] * sets

    def e2e_step(i):
        j = i % sets
        for u, up in enumerate(ups):
            if started[j]:
                up.wait_event(consumed[j])
            with torch.cuda.stream(up):
                for n in names:
                    if up_of[n] == u:
                        dev[j][n].copy_(host[n], non_blocking=True)
            loaded[j][u].record(up)
            stream.wait_event(loaded[j][u])
        if started[j]:
            stream.wait_event(fetched[j])
        o, hT = outs[j]
        d = dev[j]
        kla.kla_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["eta"], inp["eps"], None, o, hT, ws,
                          case.chunk, stream)
        consumed[j].record(stream)
        down.wait_event(consumed[j])
        with torch.cuda.stream(down):
            outs_h[j][0].copy_(o, non_blocking=True)
            outs_h[j][1].copy_(hT, non_blocking=True)
        fetched[j].record(down)
        started[j] = True

    Ke = max(3, min(K, 20))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    # three timed windows of Ke steps; the median window is reported, so that
    # one stall of the host (another process, the clock sampler) does not set it
    windows = []
    for w in range(3):
        barrier()
        t0 = time.perf_counter()
        for i in range(Ke):
            e2e_step(i)
        torch.cuda.synchronize()
        windows.append((time.perf_counter() - t0) / Ke)
    e2e_job, e2e_s = job_throughput(work["tokens"], sorted(windows)[1])
    assert kla.kla_workspace_check(ws, stream) == kla.KLA_OK
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0])
    return dict(value=e2e_job, unit="tokens/s", h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                ms_per_step=e2e_s * 1e3, steps=Ke, windows=3,
                pipeline=f"{sets} device buffer sets; H2D of step i+1 ({up_streams} copy streams) and D2H "
                         "of step i-1 overlap step i; median of 3 timed windows")


def bench_backward(case, K, W, flush, peaks, stream):
    """Time kla_chunk_bwd (the gradients of o and hT w.r.t. every input) on ``case``."""
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(case, device="cuda")
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    gen = torch.Generator(device="cuda")
    gen.manual_seed(case.seed + 1000)
    do = torch.randn((B, T, H, dv), generator=gen, device="cuda").to(inp["q"].dtype)
    dhT = torch.randn((B, H, dk, dv), generator=gen, device="cuda")
    io = kla.KLA_IO_BF16 if case.io == "bf16" else kla.KLA_IO_FP32
    ws = torch.empty(kla.kla_chunk_bwd_workspace_bytes(B, T, H, dk, dv, case.chunk, io),
                     dtype=torch.uint8, device="cuda")
    gq, gk, gv = torch.empty_like(inp["q"]), torch.empty_like(inp["k"]), torch.empty_like(inp["v"])
    gg, ge = torch.empty_like(inp["g"]), torch.empty_like(inp["eta"])
    gh0 = torch.empty_like(dhT)

    def step():
        kla.kla_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"], inp["h0"],
                          do, dhT, gq, gk, gv, gg, ge, gh0, ws, stream=stream)

    barrier()
    ms = timed_steps(step, K, W, flush, stream)
    barrier()
    work = backward_work(case)
    _, slowest_s = job_throughput(work["tokens"], sum(ms) / len(ms) * 1e-3)
    mean_ms = slowest_s * 1e3
    res = dict(ms_per_step=mean_ms, tokens_per_s=work["tokens"] / (mean_ms * 1e-3),
               roofline=dict(roofline(work, mean_ms * 1e-3, peaks, TRAFFIC_BYTES.get("bwd_" + case.name)),
                             scope="one kla_chunk_bwd call: its three launches (prep, the two carries in one grid, gradients)"),
               launches=3 * K, min_ms=min(ms), workspace_bytes=ws.numel())
    del inp, do, dhT, ws, gq, gk, gv, gg, ge, gh0
    return res


def deltakata_work(case, p):
    """Algorithmic bytes of one DeltaKATA prefill from raw inputs: q, k with p
    values per token-head, v and o with dv, g and eta; hT per head."""
    esz = 2 if case.io == "bf16" else 4
    th = case.B * case.T * case.H
    per_tok = esz * (2 * p + 2 * case.dv) + 8
    w = prefill_work(case)
    return dict(bytes=th * per_tok + case.B * case.H * case.dk * case.dv * 4, flops=w["flops"],
                tokens=case.B * case.T, token_heads=th, per_token_head_bytes=per_tok)


def bench_deltakata(case, p, K, W, flush, peaks, stream):
    """Time DeltaKATA on ``case`` from q, k with p values per token-head:
    kla_deltakata_fwd, which forms the case.dk PSD features inside the prefill
    (or, for a shape it does not take, kla_psd_features of q and k and then
    kla_chunk_fwd on them)."""
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(case, device="cuda")
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    gen = torch.Generator(device="cuda")
    gen.manual_seed(case.seed + 2000)
    dt = inp["q"].dtype
    q = torch.randn((B, T, H, p), generator=gen, device="cuda").mul(0.4).to(dt)
    u = torch.randn((B, T, H, p), generator=gen, device="cuda")
    k = (u / u.norm(dim=-1, keepdim=True)).to(dt)
    o = torch.empty((B, T, H, dv), dtype=dt, device="cuda")
    hT = torch.empty((B, H, dk, dv), dtype=torch.float32, device="cuda")
    io = kla.KLA_IO_BF16 if case.io == "bf16" else kla.KLA_IO_FP32
    n_fused = kla.kla_deltakata_fwd_workspace_bytes(B, T, H, p, dv, case.chunk, io) if dk == 128 else 0
    if n_fused:
        ws = torch.empty(n_fused, dtype=torch.uint8, device="cuda")

        def step():
            kla.kla_deltakata_fwd(q, k, inp["v"], inp["g"], inp["eta"], inp["eps"], None, o, hT, ws,
                                  chunk=case.chunk, stream=stream)
        scope, launches = "one kla_deltakata_fwd call (features formed in the prep lanes)", prefill_launches(kla, case)
    else:
        fq = torch.empty((B, T, H, dk), dtype=dt, device="cuda")
        fk = torch.empty_like(fq)
        ws = kla.alloc_workspace(B, T, H, dk, dv, case.chunk, io)

        def step():
            kla.kla_psd_features(q, fq, stream)
            kla.kla_psd_features(k, fk, stream)
            kla.kla_chunk_fwd(fq, fk, inp["v"], inp["g"], inp["eta"], inp["eps"], None, o, hT, ws,
                              case.chunk, stream)
        scope, launches = "two kla_psd_features calls and one kla_chunk_fwd call", 2 + prefill_launches(kla, case)

    barrier()
    ms = timed_steps(step, K, W, flush, stream)
    barrier()
    work = deltakata_work(case, p)
    _, slowest_s = job_throughput(work["tokens"], sum(ms) / len(ms) * 1e-3)
    mean_ms = slowest_s * 1e3
    res = dict(ms_per_step=mean_ms, tokens_per_s=work["tokens"] / (mean_ms * 1e-3),
               roofline=dict(roofline(work, mean_ms * 1e-3, peaks, TRAFFIC_BYTES.get("deltakata_" + case.name)),
                             scope=scope),
               launches=K * launches)
    del inp, q, k, o, hT, ws
    return res


def loglinear_work(case, L):
    """Algorithmic bytes of one kla_loglinear_fwd call: q, k, v, o, g, eta and
    the L level weights once per token-head.  Flops: those of the plain
    prefill (a lower bound; the level states add O(log T) per chunk)."""
    w = prefill_work(case)
    th = case.B * case.T * case.H
    per_tok = w["per_token_head_bytes"] + 4 * L
    return dict(bytes=th * per_tok, flops=w["flops"], tokens=case.B * case.T, token_heads=th,
                per_token_head_bytes=per_tok)


def bench_loglinear(case, K, W, flush, peaks, stream):
    """Time kla_loglinear_fwd on ``case`` with random level weights."""
    import chunked_delta_rule_kla_gb300 as kla
    inp = kla_inputs.make_prefill(case, device="cuda")
    B, T, H, dk, dv = case.B, case.T, case.H, case.dk, case.dv
    L = kla.kla_loglinear_num_levels(T)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(case.seed + 3000)
    lam = torch.empty((B, T, H, L), device="cuda").uniform_(0.2, 1.5, generator=gen)
    o = torch.empty((B, T, H, dv), dtype=inp["q"].dtype, device="cuda")
    io = kla.KLA_IO_BF16 if case.io == "bf16" else kla.KLA_IO_FP32
    ws = torch.empty(kla.kla_loglinear_workspace_bytes(B, T, H, dk, dv, case.chunk, io),
                     dtype=torch.uint8, device="cuda")

    def step():
        kla.kla_loglinear_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], lam, inp["eps"], o,
                              ws, stream=stream)

    barrier()
    ms = timed_steps(step, K, W, flush, stream)
    barrier()
    work = loglinear_work(case, L)
    _, slowest_s = job_throughput(work["tokens"], sum(ms) / len(ms) * 1e-3)
    mean_ms = slowest_s * 1e3
    res = dict(ms_per_step=mean_ms, tokens_per_s=work["tokens"] / (mean_ms * 1e-3), levels=L,
               roofline=dict(roofline(work, mean_ms * 1e-3, peaks, TRAFFIC_BYTES.get("loglinear_" + case.name)),
                             scope="one kla_loglinear_fwd call: its four launches (chunk records, in-chunk levels, "
                                   "one carry pass per level above the chunk, bf16 conversion)"),
               launches=4 * K, min_ms=min(ms))
    del inp, lam, o, ws
    return res


def loglinear_decode_bytes(B, H, dk, dv, L, steps, esz):
    """Algorithmic bytes of Log-Linear decoding tokens 0 .. steps-1: at token
    t > 0, with b the lowest set bit of t, each non-empty level is read
    (popcount(t-1) + 1 of them), the levels above b + 1 are written back, and
    the merged level b + 1 and the new level 0 are written; plus each token's
    q, k, v, o, g, eta and lambda."""
    sbytes = dk * dv * 4
    total = 0
    for t in range(steps):
        touched = 0
        if t > 0:
            present = bin(t - 1).count("1") + 1
            b = (t & -t).bit_length() - 1          # levels 0 .. b merge into b + 1
            touched = present * sbytes + (present - (b + 1)) * sbytes + sbytes
        total += B * H * (touched + sbytes + esz * (2 * dk + 2 * dv) + 8 + 4 * L)
    return total


def bench_loglinear_decode(case, steps, peaks, stream):
    """Time kla_loglinear_decode_step over tokens 0 .. steps-1 of ``case``'s
    heads (states zero at token 0).  Algorithmic bytes of token t > 0, with b
    the lowest set bit of t: each non-empty bucket state read (popcount(t-1)
    + 1 of them), those above level b + 1 written back, the merged level b + 1
    and the new level 0 written; q, k, v, o, g, eta, lambda."""
    import chunked_delta_rule_kla_gb300 as kla
    B, H, dk, dv = case.B, case.H, case.dk, case.dv
    L = kla.kla_loglinear_num_levels(steps)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(case.seed + 4000)
    dt = torch.bfloat16 if case.io == "bf16" else torch.float32
    q = torch.randn((steps, B, H, dk), generator=gen, device="cuda").to(dt)
    k = torch.nn.functional.normalize(torch.randn((steps, B, H, dk), generator=gen, device="cuda"), dim=-1).to(dt)
    v = torch.randn((steps, B, H, dv), generator=gen, device="cuda").to(dt)
    g = torch.nn.functional.logsigmoid(torch.randn((steps, B, H), generator=gen, device="cuda") + 2.0)
    eta = torch.sigmoid(torch.randn((steps, B, H), generator=gen, device="cuda"))
    lam = torch.empty((steps, B, H, L), device="cuda").uniform_(0.2, 1.5, generator=gen)
    states = torch.zeros((B, H, L, dk, dv), device="cuda")
    o = torch.empty((B, H, dv), dtype=dt, device="cuda")
    esz = 2 if case.io == "bf16" else 4
    total = loglinear_decode_bytes(B, H, dk, dv, L, steps, esz)

    def run():
        for t in range(steps):
            kla.kla_loglinear_decode_step(q[t], k[t], v[t], g[t], eta[t], lam[t], 1e-6, states, t, o,
                                          stream=stream)

    states.zero_()
    run()                                   # warm-up pass
    states.zero_()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    sec = e0.elapsed_time(e1) * 1e-3
    work = dict(bytes=total / steps, flops=0)    # per call, averaged over the calls
    res = dict(us_per_step=sec / steps * 1e6, tokens_per_s=B * steps / sec, levels=L,
               roofline=dict(roofline(work, sec / steps, peaks),
                             scope=f"{steps} kla_loglinear_decode_step calls from token 0, averaged"),
               launches=steps)
    del q, k, v, g, eta, lam, states, o
    return res


def bench_decode(case, K_loops, W_loops, peaks, stream, n_states=4, e2e=True):
    """Times `steps` consecutive kla_decode_step calls per loop.  The calls
    rotate over n_states independent state buffers (like the layers of a
    model), so the state working set (n_states x 64 MiB) exceeds L2."""
    import chunked_delta_rule_kla_gb300 as kla
    steps = case.steps
    inp = kla_inputs.make_decode(case, device="cuda")
    states = [inp["S"].clone() for _ in range(n_states)]
    o = torch.empty((case.B, case.H, case.dv), dtype=inp["q"].dtype, device="cuda")

    def loop():
        for t in range(steps):
            kla.kla_decode_step(inp["q"][t], inp["k"][t], inp["v"][t], inp["g"][t], inp["eta"][t],
                                inp["eps"], states[t % n_states], o, stream)

    barrier()
    ms = timed_steps(loop, K_loops, W_loops, None, stream)
    barrier()
    work = decode_work(case)
    per_call_s = max_over_ranks(sum(ms) / len(ms) / steps * 1e-3)
    res = dict(ms_per_call=per_call_s * 1e3, tokens_per_s=work["tokens"] / per_call_s,
               gbps=work["bytes"] / per_call_s / 1e9,
               roofline=dict(roofline(work, per_call_s, peaks, TRAFFIC_BYTES.get(case.name)),
                             scope="one kla_decode_step call (decode_tma_kernel)"),
               work=work, launches=K_loops * steps * LAUNCHES_PER_DECODE, calls_per_loop=steps,
               states_rotated=n_states)

    if not e2e:
        del inp, states
        return res
    # end to end: per call, pinned host q/k/v/g/eta -> device, step, o -> host
    hq = {n: inp[n][:64].cpu().pin_memory() for n in ("q", "k", "v", "g", "eta")}
    dq = {n: torch.empty_like(hq[n][0], device="cuda") for n in hq}
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    n_e2e = 64
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for t in range(n_e2e):
        for n in hq:
            dq[n].copy_(hq[n][t], non_blocking=True)
        kla.kla_decode_step(dq["q"], dq["k"], dq["v"], dq["g"], dq["eta"], inp["eps"],
                            states[t % n_states], o, stream)
        o_h.copy_(o, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e)
    res["e2e"] = dict(value=case.B / e2e_s, unit="tokens/s",
                      h2d_bytes_per_step=sum(t[0].numel() * t.element_size() for t in hq.values()),
                      d2h_bytes_per_step=o_h.numel() * o_h.element_size(), ms_per_step=e2e_s * 1e3)
    del inp, states
    return res


def cpu_baseline_prefill(case, max_heads=64):
    """The fp64 oracle as it stands, on the host cores, on a bounded sample:
    the first `max_heads` heads of the workload over the full sequence."""
    import oracle
    inp = kla_inputs.make_prefill(case.with_(B=1, H=max_heads), device="cpu")
    cores = os.cpu_count() or 1
    threads = min(cores, max_heads)
    t0 = time.perf_counter()
    oracle.kla_oracle_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["eta"], inp["eps"],
                              inp["h0"], threads=threads)
    dt = time.perf_counter() - t0
    th = case.T * max_heads
    tokens_equiv = th / case.H  # tokens of the workload whose all H heads this sample covers
    return dict(value=tokens_equiv / dt, unit="tokens/s", cores=threads, kind="oracle",
                sample=f"{max_heads} heads x T={case.T} of {case.name} ({th} token-heads), "
                       f"{dt:.2f} s wall, fp64 sequential loop, one thread per head")


# ------------------------------------------------------------------- main

def run_reference(args, rank):
    if rank != 0:
        return
    case = kla_inputs.TRAIN
    per = []
    for _ in range(args.warmup):
        cpu_baseline_prefill(case, max_heads=args.ref_heads)
    for _ in range(args.steps):
        per.append(cpu_baseline_prefill(case, max_heads=args.ref_heads))
    val = statistics.median(p["value"] for p in per)
    line = dict(impl="reference", metric=METRIC, value=val, unit="tokens/s", n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=case.B * case.T / val * 1e3,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=dict(workload=case.name, B=case.B, T=case.T, H=case.H,
                                              dk=case.dk, dv=case.dv, chunk=case.chunk),
                cpu_baseline=dict(per[0], value=val),
                e2e=dict(value=val, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-secondary", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-heads", type=int, default=64)
    ap.add_argument("--decode-loops", type=int, default=3)
    ap.add_argument("--only", choices=["train", "long", "gdn", "decode", "bwd", "deltakata", "loglinear",
                                       "lldecode"],
                    default=None,
                    help="time one workload only (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    import chunked_delta_rule_kla_gb300 as kla
    kla.load_library()
    peaks = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    clocks = ClockSampler(torch.cuda.current_device()).start()

    e2e = not args.no_e2e
    if args.only is not None:
        if args.only == "lldecode":
            dr2 = bench_loglinear_decode(kla_inputs.DECODE, 1024, peaks, stream)
            line = dict(workload="loglinear_decode_bf16_B64H16d128_x1024", tokens_per_s=dr2["tokens_per_s"],
                        us_per_step=dr2["us_per_step"], roofline=dr2["roofline"],
                        gpu_launches=dr2["launches"])
        elif args.only == "loglinear":
            lr2 = bench_loglinear(kla_inputs.TRAIN, args.steps, args.warmup, flush, peaks, stream)
            line = dict(workload="loglinear_" + kla_inputs.TRAIN.name, tokens_per_s=lr2["tokens_per_s"],
                        ms_per_step=lr2["ms_per_step"], roofline=lr2["roofline"],
                        gpu_launches=lr2["launches"])
        elif args.only == "deltakata":
            kr = bench_deltakata(kla_inputs.TRAIN, 15, args.steps, args.warmup, flush, peaks, stream)
            line = dict(workload="deltakata_p15_" + kla_inputs.TRAIN.name, tokens_per_s=kr["tokens_per_s"],
                        ms_per_step=kr["ms_per_step"], roofline=kr["roofline"],
                        gpu_launches=kr["launches"])
        elif args.only == "bwd":
            br = bench_backward(kla_inputs.TRAIN, args.steps, args.warmup, flush, peaks, stream)
            line = dict(workload="bwd_" + kla_inputs.TRAIN.name, tokens_per_s=br["tokens_per_s"],
                        ms_per_step=br["ms_per_step"], roofline=br["roofline"],
                        gpu_launches=br["launches"])
        elif args.only == "decode":
            dr = bench_decode(kla_inputs.DECODE, args.decode_loops, args.warmup, peaks, stream, e2e=e2e)
            line = dict(workload=kla_inputs.DECODE.name, tokens_per_s=dr["tokens_per_s"],
                        us_per_call=dr["ms_per_call"] * 1e3, roofline=dr["roofline"],
                        gpu_launches=dr["launches"])
        else:
            case = {"train": kla_inputs.TRAIN, "long": kla_inputs.LONG,
                    "gdn": kla_inputs.GDN_TRAIN}[args.only]
            r = bench_prefill(case, args.steps, args.warmup, flush, peaks, stream, e2e=e2e,
                              direct=args.only == "gdn")
            line = dict(workload=case.name, tokens_per_s=r["tokens_per_s"], ms_per_step=r["ms_per_step"],
                        roofline=r["roofline"], gpu_launches=r["launches"], e2e=r.get("e2e"))
        clocks.stop()
        if rank == 0:
            print(json.dumps(dict(only=args.only, **line)), flush=True)
        return
    main_case = kla_inputs.TRAIN
    head = bench_prefill(main_case, args.steps, args.warmup, flush, peaks, stream, e2e=e2e)
    secondary = {}

    def compact(r, **extra):
        rf = {k: r["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        return dict(extra, ms_per_step=round(r["ms_per_step"], 5), tokens_per_s=round(r["tokens_per_s"]),
                    roofline=rf)

    if not args.no_secondary:
        # The rows beyond the hot path first; the long prefill and the decode
        # step (the metric's other two workloads) close the line.
        gc = kla_inputs.GDN_TRAIN
        gr = bench_prefill(gc, max(5, args.steps // 2), 3, flush, peaks, stream, e2e=False,
                           direct=True)
        secondary["gdn_train_prefill"] = compact(gr, workload=gc.name, beta="direct")
        br = bench_backward(kla_inputs.TRAIN, max(5, args.steps // 4), 3, flush, peaks, stream)
        secondary["backward_train"] = compact(br, workload="bwd_" + kla_inputs.TRAIN.name)
        kr = bench_deltakata(kla_inputs.TRAIN, 15, max(5, args.steps // 2), 3, flush, peaks, stream)
        secondary["deltakata_train_prefill"] = compact(kr, workload="deltakata_p15_" + kla_inputs.TRAIN.name)
        lr2 = bench_loglinear(kla_inputs.TRAIN, max(5, args.steps // 4), 3, flush, peaks, stream)
        secondary["loglinear_train_prefill"] = compact(lr2, workload="loglinear_" + kla_inputs.TRAIN.name,
                                                       levels=lr2["levels"])
        dr2 = bench_loglinear_decode(kla_inputs.DECODE, 1024, peaks, stream)
        rf = {k: dr2["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
        secondary["loglinear_decode"] = dict(workload="loglinear_decode_bf16_B64H16d128_x1024",
                                             us_per_step=round(dr2["us_per_step"], 2),
                                             tokens_per_s=round(dr2["tokens_per_s"]), roofline=rf)
        lc = kla_inputs.LONG
        lr = bench_prefill(lc, max(3, args.steps // 10), 3, flush, peaks, stream, e2e=e2e)
        secondary["long_prefill"] = dict(compact(lr, workload=lc.name, segments=lr["segments"]),
                                         e2e=lr.get("e2e"))
        dc = kla_inputs.DECODE
        dr = bench_decode(dc, args.decode_loops, 3, peaks, stream, e2e=e2e)
        rf = {k: dr["roofline"][k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
        secondary["decode"] = dict(workload=dc.name, us_per_call=round(dr["ms_per_call"] * 1e3, 3),
                                   tokens_per_s=round(dr["tokens_per_s"]), hbm_gbs=round(dr["gbps"], 1),
                                   roofline=rf, e2e=dr.get("e2e"))
    clk = clocks.stop()
    if rank != 0:
        return
    n = world
    line = dict(
        metric=METRIC, value=head["job_tokens_per_s"], unit="tokens/s", n_gpus=n,
        steps=args.steps, warmup=args.warmup, ms_per_step=head["ms_per_step"],
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
        data="synthetic",
        config=dict(workload=main_case.name, B=main_case.B, T=main_case.T, H=main_case.H,
                    dk=main_case.dk, dv=main_case.dv, chunk=main_case.chunk),
        run=dict(io="bf16", l2="flushed between timed steps (512 MiB write, outside the events)",
                 parallelism=f"replicas x{n}" if n > 1 else "single GPU"),
        tflops=head["tflops"], hbm_gbs_algorithmic=head["gbps"],
        roofline=head["roofline"],
        e2e=head.get("e2e"),
        gpu_launches=head["launches"], clocks=clk,
    )
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(main_case, max_heads=args.ref_heads)
    line["secondary"] = secondary
    print(json.dumps(line), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
