#!/usr/bin/env python
"""Benchmark: window + landmark sparse attention forward on GB300.

One step = one pass of the hot path over one layer of synthetic input:
landmark pooling (K1) then the fused window + landmark attention (K2) on the
128K-token 70B-style layer (n=131072, 64 query / 8 KV heads, d=128, w=4096,
512 landmarks, bf16).  The headline value is useful TFLOP/s of that step
(4 * d * Hq * sum_i |attended set of row i|; masked work not counted).
The same run also measures the other configurations -- the 2K fp32 case
(CUDA-core kernel), the 32K layer with outlier keys, the million-token
layer, the Ring Attention emulation (8 KV-chunk partials + LSE merge, K3)
-- and the pattern variants and backward, under "also".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl msa|reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step on one GPU); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "128k_70b_layer"
METRIC = "sparse-attn fwd TFLOP/s & tokens/s at 128K and 1M tokens; % of bf16 TC peak"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# DRAM traffic of one attention launch on the 128K layer, from the
# committed ncu capture of this kernel.  It only applies to the kernel
# source it was measured on (SHA-256 of the attention kernel's sources);
# after any change the traffic is reported as null.
ATTN_TRAFFIC = {"128k_70b_layer": {
    "bytes": 4 * (672.524032e6 + 507.684864e6),  # the 32K capture, scaled by n
    "kernel_sha256": "1e0c40a0ab7c324000a3459add74a9af9d38bd2eab99a186c9dfae4a5cbbee51"}}


def kernel_sha256() -> str:
    """SHA-256 over the attention kernel's source and the headers it
    includes: recorded DRAM traffic is reported only for this exact code."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "long_context_sparse_landmark_gb300", "csrc")
    for name in ("k2_attn_tc2.cu", "tc_pair.cuh", "tc_ptx.cuh", "tc_sync.cuh", "tma_map.h",
                 "msa_common.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def attn_traffic(name: str):
    rec = ATTN_TRAFFIC.get(name)
    if not rec or rec["bytes"] is None or rec["kernel_sha256"] != kernel_sha256():
        return None
    return rec["bytes"]


def attended_total(wl) -> int:
    """sum_i |window(i)| + |visible landmarks(i)| for one head (closed form)."""
    import numpy as np
    i = np.arange(wl.n, dtype=np.int64)
    win = np.minimum(wl.window, i + 1).sum()
    lm = np.clip((i - wl.window + 1) // wl.block, 0, wl.G).sum() if wl.G else 0
    return int(win + lm)


def useful_flops(wl) -> float:
    return 4.0 * wl.d * wl.Hq * attended_total(wl)


def reduce_max(value: float, dist, device) -> float:
    """Maximum of a per-rank timing over all ranks (the slowest replica sets
    the job's time); identity without a process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, ms_per_step: float) -> float:
    """Whole-job units per second: every rank processes units_per_rank per
    step (weak scaling) and the step takes the slowest rank's time."""
    return world * units_per_rank / (ms_per_step * 1e-3)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
# L2 of a GB300 is 129 MB (nominal): a workload whose inputs are smaller than
# twice that has the L2 flushed (a 512 MB write) before each timed step.
L2_BYTES = 129 * 10**6
FLUSH_BYTES = 512 << 20


def run_window_landmark(wl, steps, warmup, dev, B, torch):
    """Device-resident inputs; each step = pool (K1) + fused attention (K2).
    Step times are taken from each step's own events, so that an L2 flush
    between steps (small workloads) stays outside them."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    scratch = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
               if in_bytes < 2 * L2_BYTES else None)
    k_lm = torch.empty((wl.G, wl.Hkv, wl.d), dtype=k.dtype, device=dev)
    v_lm = torch.empty_like(k_lm)
    out = torch.empty((wl.n, wl.Hq, wl.d), dtype=q.dtype, device=dev)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        B.landmark_pool(k, v, k_lm, v_lm, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(warmup):
        if scratch is not None:
            scratch.zero_()
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        if scratch is not None:
            scratch.zero_()  # evicts the inputs from L2, outside the step's events
        step(evs[s])
    t1.record(stream)
    torch.cuda.synchronize()
    assert B.device_status() == 0, "a bounded device wait ran out"
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    total_ms = sum(step_ms) if scratch is not None else t0.elapsed_time(t1)
    pool_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    res = {"total_ms": total_ms, "ms_per_step": total_ms / steps,
           "pool_ms": statistics.median(pool_ms), "attn_ms": statistics.median(attn_ms),
           "launches_per_step": 2,
           "l2": (f"L2 flushed before every step ({FLUSH_BYTES >> 20} MB write; inputs "
                  f"{in_bytes / 1e6:.0f} MB)" if scratch is not None else
                  f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB of Q, K, V)")}
    del q, k, v, k_lm, v_lm, out, lse, scratch
    torch.cuda.empty_cache()
    return res


def run_e2e(wl, steps, dev, torch):
    """Through the C entry point for host buffers (msa_attn_fwd_host, via
    msa_attention_host) with pinned HOST inputs and outputs: every step
    copies Q/K/V host->device, pools, runs the attention on row chunks and
    copies O and lse back, the copies overlapping the kernels; the call
    returns with the host results final."""
    import long_context_sparse_landmark_gb300 as pkg
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    del q, k, v
    torch.cuda.empty_cache()
    ho = torch.empty((wl.n, wl.Hq, wl.d), dtype=hq.dtype).pin_memory()
    hl = torch.empty((wl.Hq, wl.n), dtype=torch.float32).pin_memory()

    def step():
        pkg.msa_attention_host(hq, hk, hv, wl.window, wl.G, wl.scale, out=ho, lse=hl,
                               device=dev)

    step()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    el = time.perf_counter() - t
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    return el / steps, h2d, d2h


def run_ring(wl, steps, warmup, dev, B, torch):
    """Ring emulation: per step 8 chunk partials (K2 partial mode) + merge (K3)."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    n, Hq, d = q.shape
    P = wl.ring_chunks
    c = n // P
    o_parts = [torch.empty((n, Hq, d), dtype=torch.float32, device=dev) for _ in range(P)]
    l_parts = [torch.empty((Hq, n), dtype=torch.float32, device=dev) for _ in range(P)]
    out = torch.empty((n, Hq, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for p in range(P):
            B.attn_fwd_partial(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], o_parts[p],
                               l_parts[p], 0, p * c, wl.window, wl.scale, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        B.lse_merge(o_parts, l_parts, out, lse, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    def fused_step():
        # One ring layer with the aggregation inside every round.
        B.attn_fwd_partial(q, k[:c], v[:c], o_parts[0], l_parts[0], 0, 0, wl.window, wl.scale,
                           stream=stream)
        for p in range(1, P):
            B.attn_fwd_partial_merge(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], o_parts[0],
                                     l_parts[0], 0, p * c, wl.window, wl.scale, stream=stream)

    for _ in range(warmup):
        step()
        fused_step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for s in range(steps):
        step(evs[s])
    fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for s in range(steps):
        fev[s][0].record(stream)
        fused_step()
        fev[s][1].record(stream)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    fused_ms = statistics.median(e[0].elapsed_time(e[1]) for e in fev)
    part_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    merge_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    # Required merge bytes: every lse_p, every O_p row with finite lse_p, output.
    finite = sum(int(torch.isfinite(l).sum()) for l in l_parts)
    merge_bytes = P * n * Hq * 4 + finite * d * 4 + n * Hq * (d * 2 + 4)
    del q, k, v, o_parts, l_parts, out, lse
    torch.cuda.empty_cache()
    return {"partials_ms": part_ms, "merge_ms": merge_ms, "merge_bytes": merge_bytes,
            "fused_ms": fused_ms, "launches_per_step": P + 1}


def band_flops(wl) -> float:
    """Useful FLOPs of the block-band mask: 4*d*Hq*sum_i |band keys of i|."""
    import numpy as np
    i = np.arange(wl.n, dtype=np.int64)
    b = i // wl.band_block
    lo = np.maximum(0, (b - wl.band_half) * wl.band_block)
    hi = np.minimum(wl.n, (b + wl.band_half + 1) * wl.band_block)
    return 4.0 * wl.d * wl.Hq * float((hi - lo).sum())


def run_band(wl, steps, warmup, dev, B, torch):
    """Block-band attention, device-resident inputs; returns ms per launch."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        B.attn_fwd_band(q, k, v, out, lse, wl.band_block, wl.band_half, wl.scale, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        B.attn_fwd_band(q, k, v, out, lse, wl.band_block, wl.band_half, wl.scale, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    del q, k, v, out, lse
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / steps


def topk_flops(wl) -> float:
    """Useful FLOPs of window + top-k blocks: every row attends its window
    and min(top_k, candidates of its 128-row query block) whole blocks."""
    import numpy as np
    i = np.arange(wl.n, dtype=np.int64)
    r0 = (i // 128) * 128
    cand = np.clip((r0 - wl.window + 1) // wl.block, 0, wl.G)
    per_row = np.minimum(wl.window, i + 1) + np.minimum(wl.top_k, cand) * wl.block
    return 4.0 * wl.d * wl.Hq * float(per_row.sum())


def run_topk(wl, steps, warmup, dev, B, torch):
    """Pool K + block select + attention in one call (msa_attn_fwd_topk),
    device-resident inputs and a preallocated workspace; also times the
    selection kernel alone.  Returns ms per call of each."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    ws = torch.empty((B.topk_workspace_size(wl.n, wl.Hkv, wl.d, wl.G, wl.top_k, q.dtype),),
                     dtype=torch.uint8, device=dev)
    k_lm = torch.empty((wl.G, wl.Hkv, wl.d), dtype=k.dtype, device=dev)
    n_qb = (wl.n + 127) // 128
    sel = torch.empty((n_qb, wl.Hkv, wl.top_k), dtype=torch.int32, device=dev)
    cnt = torch.empty((n_qb, wl.Hkv), dtype=torch.int32, device=dev)
    B.landmark_pool(k, v, k_lm, torch.empty_like(k_lm))
    stream = torch.cuda.current_stream()

    def timed(fn, n_iter):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n_iter):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n_iter

    fused_ms = timed(lambda: B.attn_fwd_topk(q, k, v, out, lse, wl.window, wl.G, wl.top_k,
                                             wl.scale, ws, stream=stream), steps)
    select_ms = timed(lambda: B.block_select(q, k_lm, sel, cnt, wl.window, wl.top_k,
                                             stream=stream), steps)
    assert B.device_status() == 0
    del q, k, v, out, lse, ws, k_lm, sel, cnt
    torch.cuda.empty_cache()
    return {"fused_ms": fused_ms, "select_ms": select_ms}


def compressed_flops(wl) -> float:
    """Useful FLOPs of window + compression tokens with global rows: rows
    c*every - 1 attend i + 1 keys, the others min(w, i+1) + L(i)."""
    import numpy as np
    i = np.arange(wl.n, dtype=np.int64)
    per_row = np.minimum(wl.window, i + 1) + np.clip((i - wl.window + 1) // wl.block, 0, wl.G)
    glob = np.asarray(wl.global_rows(), dtype=np.int64)
    per_row[glob] = glob + 1
    return 4.0 * wl.d * wl.Hq * float(per_row.sum())


def run_compressed(wl, steps, warmup, dev, B, torch):
    """Compression tokens (pool with n/32 blocks) + window/compression
    attention + global rows, device-resident inputs and preallocated
    buffers; returns ms per step and of the global-rows call alone."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    k_lm = torch.empty((wl.G, wl.Hkv, wl.d), dtype=k.dtype, device=dev)
    v_lm = torch.empty_like(k_lm)
    rows = torch.as_tensor(wl.global_rows(), dtype=torch.int64, device=dev)
    ws = torch.empty((B.global_rows_workspace_size(wl.n, rows.numel(), wl.Hq, wl.Hkv, wl.d),),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        B.landmark_pool(k, v, k_lm, v_lm, stream=stream)
        B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale, stream=stream)
        B.attn_fwd_global_rows(q, k, v, rows, out, lse, wl.scale, ws, stream=stream)

    def glob():
        B.attn_fwd_global_rows(q, k, v, rows, out, lse, wl.scale, ws, stream=stream)

    res = {}
    for name, fn in (("step_ms", step), ("global_ms", glob)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / steps
    assert B.device_status() == 0
    del q, k, v, out, lse, k_lm, v_lm, ws
    torch.cuda.empty_cache()
    return res


def run_bwd(wl, steps, warmup, dev, B, torch):
    """Backward of the window + landmark layer (msa_attn_bwd) on device-
    resident q, k, v, out, lse, dout and preallocated gradients; returns ms
    per call."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    k_lm = torch.empty((wl.G, wl.Hkv, wl.d), dtype=k.dtype, device=dev)
    v_lm = torch.empty_like(k_lm)
    out = torch.empty_like(q)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    B.landmark_pool(k, v, k_lm, v_lm)
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    dout = torch.randn(q.shape, generator=gen, device=dev).to(torch.bfloat16)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = torch.empty((B.attn_bwd_workspace_size(wl.n, wl.Hq, wl.Hkv, wl.d, wl.G),),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        B.attn_bwd(q, k, v, k_lm, v_lm, out, lse, dout, dq, dk, dv, wl.window, wl.G, wl.scale,
                   ws, stream=stream)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    del q, k, v, out, lse, dout, dq, dk, dv, ws, k_lm, v_lm
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / steps


def run_bwd_compressed(wl, steps, warmup, dev, B, torch):
    """Backward of the compression-token pattern (msa_attn_bwd_global_rows)
    on device-resident tensors; returns ms per call."""
    from long_context_sparse_landmark_gb300.workloads import generate
    q, k, v = generate(wl, device=dev)
    k_lm = torch.empty((wl.G, wl.Hkv, wl.d), dtype=k.dtype, device=dev)
    v_lm = torch.empty_like(k_lm)
    out = torch.empty_like(q)
    lse = torch.empty((wl.Hq, wl.n), dtype=torch.float32, device=dev)
    rows = torch.as_tensor(wl.global_rows(), dtype=torch.int64, device=dev)
    fws = torch.empty((B.global_rows_workspace_size(wl.n, rows.numel(), wl.Hq, wl.Hkv, wl.d),),
                      dtype=torch.uint8, device=dev)
    B.landmark_pool(k, v, k_lm, v_lm)
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale)
    B.attn_fwd_global_rows(q, k, v, rows, out, lse, wl.scale, fws)
    del fws
    gen = torch.Generator(device=dev)
    gen.manual_seed(8)
    dout = torch.randn(q.shape, generator=gen, device=dev).to(torch.bfloat16)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ws = torch.empty((B.attn_bwd_global_rows_workspace_size(wl.n, rows.numel(), wl.Hq, wl.Hkv,
                                                            wl.d, wl.G),),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def call():
        B.attn_bwd_global_rows(q, k, v, k_lm, v_lm, out, lse, dout, rows, dq, dk, dv, wl.window,
                               wl.G, wl.scale, ws, stream=stream)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    del q, k, v, out, lse, dout, dq, dk, dv, ws, k_lm, v_lm
    torch.cuda.empty_cache()
    return e0.elapsed_time(e1) / steps


def fp32_fma_peak_tflops(torch, sm_max_mhz=None) -> float:
    """FP32 FMA peak of the GPU: SMs x 128 FP32 lanes x 2 FLOP per fused
    multiply-add x the maximum SM clock (GB300: 152 x 128 x 2 x 2.07 GHz)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    mhz = sm_max_mhz or 2070.0
    return sms * 128 * 2 * mhz * 1e6 / 1e12


def cpu_baseline(wl, rows_target, torch):
    """The fp64 oracle on the host cores, on a bounded row sample of the
    same workload; extrapolated to the full layer by rows."""
    import numpy as np
    import oracle
    from long_context_sparse_landmark_gb300.workloads import generate, to_numpy_bits
    oracle.set_threads(os.cpu_count() or 1)
    q, k, v = generate(wl, device="cuda")
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(wl.n, size=rows_target, replace=False)).astype(np.int64)
    qs = to_numpy_bits(q.index_select(0, torch.as_tensor(rows, device=q.device)))
    kn, vn = to_numpy_bits(k), to_numpy_bits(v)
    del q, k, v
    torch.cuda.empty_cache()
    t = time.perf_counter()
    k_lm = oracle.landmark_pool(kn, wl.G)
    v_lm = oracle.landmark_pool(vn, wl.G)
    pool_s = time.perf_counter() - t
    t = time.perf_counter()
    oracle.attn(qs, kn, vn, wl.window, wl.G, wl.scale, q_positions=rows, landmarks=(k_lm, v_lm))
    rows_s = time.perf_counter() - t
    cores = oracle.get_threads()

    def flops_of(r):
        per_row = np.minimum(wl.window, r + 1) + np.clip((r - wl.window + 1) // wl.block, 0, wl.G)
        return 4.0 * wl.d * wl.Hq * float(per_row.sum())

    full_s = pool_s + rows_s * useful_flops(wl) / flops_of(rows)
    # The same oracle on one thread, on the first 1/16 of the sample.
    r1 = rows[: max(1, rows_target // 16)]
    oracle.set_threads(1)
    t = time.perf_counter()
    oracle.attn(qs[: len(r1)], kn, vn, wl.window, wl.G, wl.scale, q_positions=r1,
                landmarks=(k_lm, v_lm))
    one_s = time.perf_counter() - t
    oracle.set_threads(cores)
    return {"value": useful_flops(wl) / full_s / 1e12, "unit": "TFLOP/s",
            "cores": cores, "kind": "oracle",
            "sample": (f"{rows_target} random rows x {wl.Hq} heads of {wl.name} "
                       f"({rows_s:.1f} s) + landmark pooling of the full K/V ({pool_s:.1f} s); "
                       f"extrapolated to all {wl.n} rows by attended keys"),
            "value_1_thread": flops_of(r1) / one_s / 1e12,
            "sample_1_thread": f"{len(r1)} of those rows on one thread ({one_s:.1f} s)",
            "wall_s": pool_s + rows_s + one_s}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--cpu-rows", type=int, default=4096)
    ap.add_argument("--workload", default=HEADLINE,
                    help="window+landmark workload timed as the step (profiling uses smaller ones)")
    ap.add_argument("--n", type=int, default=None,
                    help="tokens of the timed step's workload, landmark block size kept "
                         "(a smaller case of the same kernel, for profiling)")
    ap.add_argument("--only", choices=["ring", "bwd", "topk"], default=None,
                    help="run only one leg: the ring emulation (partials, merge, fused "
                         "rounds), the backward pass, or the top-k call (for profiling)")
    ap.add_argument("--leg-n", type=int, default=None,
                    help="tokens of the --only bwd / topk leg (default: the workload's)")
    ap.add_argument("--ring-n", type=int, default=None,
                    help="tokens of the ring emulation (default 131072; smaller for profiling)")
    ap.add_argument("--no-also", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    import torch
    from long_context_sparse_landmark_gb300.workloads import WORKLOADS
    wl = WORKLOADS[args.workload]
    if args.n:
        wl = wl.with_n(args.n, G=args.n // wl.block if wl.G else 0,
                       name=f"{wl.name}_n{args.n}")
    peaks = load_peaks()

    if args.impl == "reference":
        run_reference(args, wl, rank, world, torch)
        return

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    from long_context_sparse_landmark_gb300 import _binding as B

    if args.only in ("bwd", "topk"):
        base = wl if args.only == "bwd" else WORKLOADS["topk_128k"]
        wlx = base.with_n(args.leg_n, name=f"{base.name}_{args.leg_n}") if args.leg_n else base
        if args.only == "bwd":
            ms = run_bwd(wlx, args.steps, args.warmup, dev, B, torch)
            res = {"workload": wlx.name, "bwd_ms": round(ms, 4),
                   "tflops": round(2.5 * useful_flops(wlx) / (ms * 1e-3) / 1e12, 2)}
        else:
            r = run_topk(wlx, args.steps, args.warmup, dev, B, torch)
            res = {"workload": wlx.name, "fused_ms": round(r["fused_ms"], 4),
                   "select_ms": round(r["select_ms"], 4)}
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    if args.only == "ring":
        wlr = WORKLOADS["ring_128k"]
        if args.ring_n:
            wlr = wlr.with_n(args.ring_n, name=f"ring_{args.ring_n}")
        rr = run_ring(wlr, args.steps, args.warmup, dev, B, torch)
        fr = useful_flops(wlr)
        if rank == 0:
            print(json.dumps({
                "workload": wlr.name, "n": wlr.n, "Hq": wlr.Hq, "Hkv": wlr.Hkv, "d": wlr.d,
                "chunks": wlr.ring_chunks, "partials_ms": round(rr["partials_ms"], 4),
                "partials_tflops": round(fr / (rr["partials_ms"] * 1e-3) / 1e12, 2),
                "merge_ms": round(rr["merge_ms"], 4), "merge_bytes": rr["merge_bytes"],
                "merge_gbs": round(rr["merge_bytes"] / (rr["merge_ms"] * 1e-3) / 1e9, 1),
                "fused_rounds_ms": round(rr["fused_ms"], 4)}), flush=True)
        return

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(local_rank) as clk:
        res = run_window_landmark(wl, args.steps, args.warmup, dev, B, torch)
    barrier()
    total_ms = reduce_max(res["total_ms"], dist, dev)
    ms_per_step = total_ms / args.steps
    flops = useful_flops(wl)
    value = job_throughput(world, flops, ms_per_step) / 1e12
    tokens_per_s = job_throughput(world, wl.n, ms_per_step)
    attn_tflops = flops / (res["attn_ms"] * 1e-3) / 1e12
    tensor_path = B.uses_tensor_cores(wl.Hq, wl.Hkv, wl.d, wl.torch_dtype)
    pool_bytes = 2 * wl.n * wl.Hkv * wl.d * 2 + 2 * wl.G * wl.Hkv * wl.d * 2
    # Q, K, V and the landmarks read once, O (bf16) and lse written once.
    attn_bytes = (wl.n * wl.Hq * wl.d * 2 + 2 * wl.n * wl.Hkv * wl.d * 2
                  + 2 * wl.G * wl.Hkv * wl.d * 2 + wl.n * wl.Hq * (wl.d * 2 + 4))

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": (f"synthetic (i.i.d. N(0,1) Q/K/V from seed {wl.seed}, {wl.dtype}"
                 + (", outlier keys" if wl.outliers else "") + ")"),
        "config": {"workload": wl.name, "n": wl.n, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "window": wl.window, "landmarks": wl.G, "batch": 1,
                   "step": "landmark pool + fused window/landmark attention",
                   "l2": res["l2"],
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(tokens_per_s, 1),
        "pct_bf16_peak": round(100.0 * value / world / peaks["bf16_tflops"], 2),
        "kernels_ms": {"landmark_pool": round(res["pool_ms"], 4),
                       "attn_fwd": round(res["attn_ms"], 4)},
        "roofline": ({"bound": "tensor", "kernel": "attn_tc2_kernel",
                      "achieved": round(attn_tflops, 2),
                      "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                      "frac": round(attn_tflops / peaks["bf16_tflops"], 4),
                      "peak_kind": f"bf16 burst ({peaks['source']}): a launch timed on its own",
                      "frac_of_sustained": round(attn_tflops / peaks["bf16_tflops_sustained"],
                                                 4),
                      "traffic": attn_traffic(wl.name),
                      "algorithmic_bytes": attn_bytes} if tensor_path else
                     {"bound": "alu", "kernel": "attn_simt_kernel",
                      "achieved": round(attn_tflops, 3),
                      "peak": round(fp32_fma_peak_tflops(torch), 1), "unit": "TFLOP/s",
                      "frac": round(attn_tflops / fp32_fma_peak_tflops(torch), 4),
                      "peak_kind": "FP32 FMA: SMs x 128 lanes x 2 FLOP x max SM clock",
                      "traffic": None, "algorithmic_bytes": attn_bytes}),
        "pool_roofline": {"bound": "hbm",
                          "achieved": round(pool_bytes / (res["pool_ms"] * 1e-3) / 1e9, 1),
                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(pool_bytes / (res["pool_ms"] * 1e-3) / 1e9
                                        / peaks["hbm_gbs"], 4)},
        "gpu_launches": res["launches_per_step"] * args.steps,
        "clocks": clk.summary(),
    }

    if not args.no_e2e and rank == 0:
        e2e_s, h2d, d2h = run_e2e(wl, 3, dev, torch)
        line["e2e"] = {"value": round(flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(e2e_s * 1e3, 3)}

    if not args.no_also and rank == 0:
        also = {}
        # The 2K fp32 case runs the CUDA-core kernel (fp32 FFMA arithmetic,
        # the 1e-5 path): FLOP/s against the FP32 FMA peak of the SMs.
        wlp = WORKLOADS["pr1_2k"]
        rp = run_window_landmark(wlp, 20, 3, dev, B, torch)
        fp = useful_flops(wlp)
        fp32_peak = fp32_fma_peak_tflops(torch, line["clocks"].get("sm_max_mhz"))
        also["pr1_2k"] = {
            "ms_per_step": round(rp["ms_per_step"], 4),
            "tokens_per_s": round(wlp.n / (rp["ms_per_step"] * 1e-3), 1),
            "attn_ms": round(rp["attn_ms"], 4), "pool_ms": round(rp["pool_ms"], 4),
            "attn_tflops": round(fp / (rp["attn_ms"] * 1e-3) / 1e12, 3),
            "roofline": {"bound": "alu", "kernel": "attn_simt_kernel", "unit": "TFLOP/s",
                         "achieved": round(fp / (rp["attn_ms"] * 1e-3) / 1e12, 3),
                         "peak": round(fp32_peak, 1),
                         "frac": round(fp / (rp["attn_ms"] * 1e-3) / 1e12 / fp32_peak, 4),
                         "peak_kind": "FP32 FMA: SMs x 128 lanes x 2 FLOP x max SM clock"},
            "dtype": "f32", "steps": 20, "l2": rp["l2"]}
        wl32 = WORKLOADS["32k_outliers"]
        r32 = run_window_landmark(wl32, 20, 3, dev, B, torch)
        f32k = useful_flops(wl32)
        also["32k_outliers"] = {
            "ms_per_step": round(r32["ms_per_step"], 4),
            "tokens_per_s": round(wl32.n / (r32["ms_per_step"] * 1e-3), 1),
            "tflops": round(f32k / (r32["ms_per_step"] * 1e-3) / 1e12, 2),
            "attn_ms": round(r32["attn_ms"], 4),
            "attn_tflops": round(f32k / (r32["attn_ms"] * 1e-3) / 1e12, 2),
            "pct_bf16_peak": round(100.0 * f32k / (r32["attn_ms"] * 1e-3) / 1e12
                                   / peaks["bf16_tflops"], 2),
            "steps": 20, "l2": r32["l2"]}
        wl1m = WORKLOADS["1m_70b_layer"]
        r1 = run_window_landmark(wl1m, 5, 1, dev, B, torch)  # medians of 5 at 1M
        f1 = useful_flops(wl1m)
        also["1m_70b_layer"] = {
            "ms_per_step": round(r1["ms_per_step"], 3),
            "tflops": round(f1 / (r1["ms_per_step"] * 1e-3) / 1e12, 2),
            "tokens_per_s": round(wl1m.n / (r1["ms_per_step"] * 1e-3), 1),
            "attn_tflops": round(f1 / (r1["attn_ms"] * 1e-3) / 1e12, 2),
            "pct_bf16_peak": round(100.0 * f1 / (r1["ms_per_step"] * 1e-3) / 1e12
                                   / peaks["bf16_tflops"], 2),
            "pool_gbs": round((2 * wl1m.n * wl1m.Hkv * wl1m.d * 2 + 2 * wl1m.G * wl1m.Hkv
                               * wl1m.d * 2) / (r1["pool_ms"] * 1e-3) / 1e9, 1),
            "steps": 5}
        wlb = WORKLOADS["band_128k"]
        bms = run_band(wlb, 3, 1, dev, B, torch)
        fb = band_flops(wlb)
        also["band_128k"] = {"ms_per_step": round(bms, 3),
                             "tflops": round(fb / (bms * 1e-3) / 1e12, 2),
                             "pct_bf16_peak": round(100.0 * fb / (bms * 1e-3) / 1e12
                                                    / peaks["bf16_tflops"], 2),
                             "steps": 3}
        wlt = WORKLOADS["topk_128k"]
        rt = run_topk(wlt, 3, 1, dev, B, torch)
        ft = topk_flops(wlt)
        # selection reads Q once (the block-mean keys are 1/256 of K)
        sel_bytes = wlt.n * wlt.Hq * wlt.d * 2
        also["topk_128k"] = {"ms_per_step": round(rt["fused_ms"], 3),
                             "tflops": round(ft / (rt["fused_ms"] * 1e-3) / 1e12, 2),
                             "pct_bf16_peak": round(100.0 * ft / (rt["fused_ms"] * 1e-3)
                                                    / 1e12 / peaks["bf16_tflops"], 2),
                             "select_ms": round(rt["select_ms"], 4),
                             "select_gbs": round(sel_bytes / (rt["select_ms"] * 1e-3) / 1e9,
                                                 1),
                             "launches_per_step": 3, "steps": 3}
        wlc = WORKLOADS["compress_128k"]
        rc = run_compressed(wlc, 3, 1, dev, B, torch)
        fc = compressed_flops(wlc)
        fg = 4.0 * wlc.d * wlc.Hq * float(sum(r + 1 for r in wlc.global_rows()))
        also["compress_128k"] = {"ms_per_step": round(rc["step_ms"], 3),
                                 "tflops": round(fc / (rc["step_ms"] * 1e-3) / 1e12, 2),
                                 "pct_bf16_peak": round(100.0 * fc / (rc["step_ms"] * 1e-3)
                                                        / 1e12 / peaks["bf16_tflops"], 2),
                                 "global_rows_ms": round(rc["global_ms"], 4),
                                 "global_rows_tflops": round(fg / (rc["global_ms"] * 1e-3)
                                                             / 1e12, 2),
                                 "launches_per_step": 4, "steps": 3}
        bms = run_bwd(wl, 3, 1, dev, B, torch)
        # Standard backward count: five GEMMs per attended pair (S, dP, dV,
        # dK, dQ), 2.5 x the forward's useful FLOPs.
        fbw = 2.5 * flops
        # Executed: the dK/dV kernels take S, dP, dV, dK (8 d per attended
        # pair) and the dQ kernel recomputes S and dP besides dQ (6 d):
        # 1.4 x the useful count.
        also["bwd_" + wl.name] = {"ms_per_step": round(bms, 3),
                                  "tflops": round(fbw / (bms * 1e-3) / 1e12, 2),
                                  "pct_bf16_peak": round(100.0 * fbw / (bms * 1e-3) / 1e12
                                                         / peaks["bf16_tflops"], 2),
                                  "executed_tflops": round(1.4 * fbw / (bms * 1e-3) / 1e12, 2),
                                  "launches_per_step": 5, "steps": 3}
        cms = run_bwd_compressed(wlc, 3, 1, dev, B, torch)
        fcb = 2.5 * fc
        also["bwd_compress_128k"] = {"ms_per_step": round(cms, 3),
                                     "tflops": round(fcb / (cms * 1e-3) / 1e12, 2),
                                     "pct_bf16_peak": round(100.0 * fcb / (cms * 1e-3) / 1e12
                                                            / peaks["bf16_tflops"], 2),
                                     "launches_per_step": 9, "steps": 3}
        wlr = WORKLOADS["ring_128k"]
        rr = run_ring(wlr, 10, 1, dev, B, torch)  # medians of 10
        fr = useful_flops(wlr)
        also["ring_128k"] = {
            "partials_ms": round(rr["partials_ms"], 3), "merge_ms": round(rr["merge_ms"], 3),
            "partials_tflops": round(fr / (rr["partials_ms"] * 1e-3) / 1e12, 2),
            "merge_gbs": round(rr["merge_bytes"] / (rr["merge_ms"] * 1e-3) / 1e9, 1),
            "merge_frac_hbm": round(rr["merge_bytes"] / (rr["merge_ms"] * 1e-3) / 1e9
                                    / peaks["hbm_gbs"], 4),
            "fused_rounds_ms": round(rr["fused_ms"], 3),
            "fused_rounds_tflops": round(fr / (rr["fused_ms"] * 1e-3) / 1e12, 2),
            "steps": 10}
        line["also"] = also

    if not args.no_cpu and rank == 0:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_rows, torch)

    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args, wl, rank, world, torch):
    """Reference arm: the fp64 oracle on the host cores (there is no code
    of the pages to install); each step evaluates a bounded row sample of
    the 128K layer, extrapolated to the full layer."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from long_context_sparse_landmark_gb300.workloads import generate, to_numpy_bits
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v = generate(wl, device=gen_dev)
    kn, vn = to_numpy_bits(k), to_numpy_bits(v)
    k_lm = oracle.landmark_pool(kn, wl.G)
    v_lm = oracle.landmark_pool(vn, wl.G)
    rows_per_step = 64
    rng = np.random.default_rng(0)
    flops_full = useful_flops(wl)

    def one(rows):
        qs = to_numpy_bits(q.index_select(0, torch.as_tensor(rows, device=q.device)))
        t = time.perf_counter()
        oracle.attn(qs, kn, vn, wl.window, wl.G, wl.scale, q_positions=rows,
                    landmarks=(k_lm, v_lm))
        el = time.perf_counter() - t
        per_row = np.minimum(wl.window, rows + 1) + np.clip((rows - wl.window + 1) // wl.block,
                                                            0, wl.G)
        return el, 4.0 * wl.d * wl.Hq * float(per_row.sum())

    for _ in range(args.warmup):
        one(np.sort(rng.choice(wl.n, rows_per_step, replace=False)).astype(np.int64))
    tot_s, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        el, f = one(np.sort(rng.choice(wl.n, rows_per_step, replace=False)).astype(np.int64))
        tot_s += el
        tot_f += f
    value = tot_f / tot_s / 1e12
    # ms_per_step is the measured time of one step (one row sample); the
    # time a whole layer would take at this rate is reported beside it.
    ms_per_step = tot_s / args.steps * 1e3
    layer_ms = flops_full / (value * 1e12) * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "step": f"{rows_per_step} random rows x {wl.Hq} heads of the layer",
            "full_layer_ms_extrapolated": layer_ms,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs)",
            "config": {"workload": wl.name, "n": wl.n, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                       "window": wl.window, "landmarks": wl.G, "batch": 1},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.get_threads(),
                             "kind": "oracle",
                             "sample": f"{rows_per_step} random rows x {wl.Hq} heads per step, "
                                       "landmarks pooled once; extrapolated to the full layer"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
