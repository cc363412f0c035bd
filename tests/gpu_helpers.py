"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import Workload, to_numpy_bits

# Tolerances: bf16 inputs with fp32 accumulation, and fp32 inputs.
BF16_MAX_ABS, BF16_MEAN_ABS = 1e-2, 1e-3
F32_MAX_ABS = 1e-5


# Canary guards: every output and workspace buffer of the GPU tests lives
# inside a larger allocation with GUARD_BYTES of a fixed byte pattern before
# and after it; check_guards() (run after each GPU test by conftest, and by
# the helpers after each call) fails if a kernel wrote outside its buffer.
GUARD_BYTES = 4096
GUARD_BYTE = 0xA5
_guarded: list = []


def gempty(shape, dtype=torch.float32, device="cuda"):
    """torch.empty inside a guarded allocation (16-byte aligned start)."""
    shape = tuple(shape) if not isinstance(shape, int) else (shape,)
    numel = math.prod(shape)
    nbytes = numel * torch.tensor([], dtype=dtype).element_size()
    raw = torch.empty((2 * GUARD_BYTES + nbytes,), dtype=torch.uint8, device=device)
    raw[:GUARD_BYTES].fill_(GUARD_BYTE)
    raw[GUARD_BYTES + nbytes:].fill_(GUARD_BYTE)
    _guarded.append((raw, nbytes, f"{tuple(shape)} {dtype}"))
    return raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)


def gempty_like(t):
    return gempty(t.shape, t.dtype, t.device)


def gfull(shape, value, dtype=torch.float32, device="cuda"):
    t = gempty(shape, dtype, device)
    t.fill_(value)
    return t


def gfull_like(t, value):
    return gfull(t.shape, value, t.dtype, t.device)


def gzeros(shape, dtype=torch.float32, device="cuda"):
    return gfull(shape, 0, dtype, device)


def check_guards(forget: bool = False):
    """Assert that no guard byte of any live guarded buffer changed."""
    bad = []
    for raw, nbytes, what in _guarded:
        head = raw[:GUARD_BYTES]
        tail = raw[GUARD_BYTES + nbytes:]
        nh = int((head != GUARD_BYTE).sum())
        nt = int((tail != GUARD_BYTE).sum())
        if nh or nt:
            bad.append(f"{what}: {nh} bytes before, {nt} bytes after changed")
    if forget:
        _guarded.clear()
    assert not bad, "write outside a buffer: " + "; ".join(bad)


def binding():
    from long_context_sparse_landmark_gb300 import _binding
    return _binding


def tol(dtype: str):
    if dtype == "bf16":
        return BF16_MAX_ABS, BF16_MEAN_ABS
    return F32_MAX_ABS, F32_MAX_ABS


def compare(gpu, ref, max_abs, mean_abs, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    both_ninf = np.isneginf(gpu) & np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), np.isneginf(ref)), f"{what}: -inf pattern differs"
    g = np.where(both_ninf, 0.0, gpu)
    r = np.where(both_ninf, 0.0, ref)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - r)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mean <= mean_abs, (
        f"{what}: max-abs {mx:.3e} (bar {max_abs:.0e}), mean-abs {mean:.3e} (bar {mean_abs:.0e})")
    return mx, mean


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def run_gpu_attention(q, k, v, wl: Workload, out_dtype=torch.float32):
    """Pool landmarks and run the fused attention through the C ABI."""
    B = binding()
    n, Hq, d = q.shape
    out = gempty((n, Hq, d), dtype=out_dtype, device=q.device)
    lse = gempty((Hq, n), dtype=torch.float32, device=q.device)
    if wl.G > 0:
        k_lm = gempty((wl.G, wl.Hkv, d), dtype=k.dtype, device=k.device)
        v_lm = gempty_like(k_lm)
        B.landmark_pool(k, v, k_lm, v_lm)
        check_guards()
    else:
        k_lm = v_lm = None
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale)
    check_guards()
    return out, lse


def oracle_attention(q, k, v, wl: Workload, rows=None):
    """Oracle on host copies of the same input bits (all rows or a sample)."""
    kn, vn = to_numpy_bits(k), to_numpy_bits(v)
    if rows is None:
        qn = to_numpy_bits(q)
        return oracle.attn(qn, kn, vn, wl.window, wl.G, wl.scale)
    idx = torch.as_tensor(rows, device=q.device)
    qn = to_numpy_bits(q.index_select(0, idx))
    return oracle.attn(qn, kn, vn, wl.window, wl.G, wl.scale,
                       q_positions=np.asarray(rows, dtype=np.int64))


def gather_rows(out, lse, rows):
    idx = torch.as_tensor(rows, device=out.device)
    o = out.index_select(0, idx).float().cpu().numpy()
    l = lse.index_select(1, idx).cpu().numpy()
    return o, l


def scale_of(d):
    return 1.0 / math.sqrt(d)
