"""GPU parity of compression tokens + global query rows through the C ABI,
against the fp64 oracle: msa_attn_fwd_global_rows alone (only the listed
rows are written, each equal to causal attention at its position; many key
splits, ragged M tiles, unsorted and repeated positions, both kernels), the
whole compressed pattern on small inputs, and the 128K workload in the
benchmark's launch configuration (all global rows plus a row sample)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import (WORKLOADS, Workload, generate,
                                                          sample_rows, to_numpy_bits)
from tests.gpu_helpers import binding, compare, gather_rows, gempty, gfull, tol

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = 7.25


@pytest.fixture(scope="module", autouse=True)
def _oracle_threads():
    import os
    oracle.set_threads(os.cpu_count() or 1)


def _run_global_rows(q, k, v, rows, scale):
    B = binding()
    n, Hq, d = q.shape
    out = gfull((n, Hq, d), SENTINEL, dtype=torch.float32, device=DEV)
    lse = gfull((Hq, n), SENTINEL, dtype=torch.float32, device=DEV)
    r = torch.as_tensor(rows, dtype=torch.int64, device=DEV)
    ws = gempty((B.global_rows_workspace_size(n, len(rows), Hq, k.shape[1], d),),
                dtype=torch.uint8, device=DEV)
    B.attn_fwd_global_rows(q, k, v, r, out, lse, 1.0 / np.sqrt(d), ws)
    torch.cuda.synchronize()
    return out, lse


GR_CASES = [
    # dt, d, n, Hq, Hkv, rows
    ("bf16", 128, 1000, 8, 2, [0, 1, 127, 128, 500, 999]),
    ("bf16", 128, 4096, 16, 2, "random40"),
    ("bf16", 128, 65536, 8, 1, [65535, 40000, 129]),
    ("f32", 64, 777, 4, 1, [776, 3, 300, 3]),
    ("bf16", 64, 2048, 6, 6, [2047, 1024, 0]),
    ("f32", 128, 300, 2, 1, [299]),
    ("bf16", 128, 257, 64, 8, [256, 0, 128]),
]


@pytest.mark.parametrize("dt,d,n,Hq,Hkv,rows", GR_CASES)
def test_global_rows_parity(dt, d, n, Hq, Hkv, rows):
    B = binding()
    if rows == "random40":
        rng = np.random.default_rng(n)
        rows = [int(x) for x in rng.choice(n, 39, replace=False)]
        rows.append(rows[5])  # a repeated position
    wl = Workload("gr", n, Hq, Hkv, d, 1, 0, dt, seed=n + Hq)
    q, k, v = generate(wl, device=DEV)
    out, lse = _run_global_rows(q, k, v, rows, wl.scale)
    assert B.device_status() == 0
    uniq = np.unique(rows)
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    ro, rl = oracle.attn(qn, kn, vn, n, 0, wl.scale, rows=uniq)
    go, gl = gather_rows(out, lse, uniq)
    mx, mean = tol(dt)
    compare(go, ro, mx, mean, f"global rows O {wl}")
    compare(gl, rl, mx, mean, f"global rows lse {wl}")
    # every other row untouched
    keep = np.setdiff1d(np.arange(n), uniq)
    o_rest, l_rest = gather_rows(out, lse, keep)
    assert np.all(o_rest == SENTINEL) and np.all(l_rest == SENTINEL)


def test_global_rows_invalid_position_is_reported_and_skipped():
    B = binding()
    n, Hq, Hkv, d = 512, 4, 1, 128
    for dt in ("bf16", "f32"):
        wl = Workload("grbad", n, Hq, Hkv, d, 1, 0, dt, seed=3)
        q, k, v = generate(wl, device=DEV)
        B.device_status(clear=True)
        out, lse = _run_global_rows(q, k, v, [100, n + 5, -1, 511], wl.scale)
        assert B.device_status(clear=True) == 1  # MSA_ERR_INVALID_ARG
        qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
        ro, rl = oracle.attn(qn, kn, vn, n, 0, wl.scale, rows=[100, 511])
        go, gl = gather_rows(out, lse, [100, 511])
        mx, mean = tol(dt)
        compare(go, ro, mx, mean, "valid rows beside invalid ones")
        keep = np.setdiff1d(np.arange(n), [100, 511])
        assert np.all(gather_rows(out, lse, keep)[0] == SENTINEL)


@pytest.mark.parametrize("dt,d,n,w,block,every", [("bf16", 128, 4096, 300, 32, 1024),
                                                  ("f32", 64, 2048, 100, 32, 500),
                                                  ("bf16", 64, 1024, 64, 16, 333)])
def test_compressed_small(dt, d, n, w, block, every):
    import long_context_sparse_landmark_gb300.api as api
    B = binding()
    wl = Workload("cmp", n, 8, 2, d, w, n // block, dt, seed=n + every, global_every=every)
    q, k, v = generate(wl, device=DEV)
    glob = wl.global_rows()
    out, lse = api.compressed_attention(q, k, v, w, block,
                                        torch.as_tensor(glob, dtype=torch.int64, device=DEV),
                                        wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    ro, rl = oracle.attn_compressed(to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v), w,
                                    block, glob, wl.scale)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"compressed O {wl}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"compressed lse {wl}")


@pytest.mark.large
def test_compress_128k_sampled_rows():
    import long_context_sparse_landmark_gb300.api as api
    wl = WORKLOADS["compress_128k"]
    q, k, v = generate(wl, device=DEV)
    glob = wl.global_rows()
    out, lse = api.compressed_attention(q, k, v, wl.window, wl.block,
                                        torch.as_tensor(glob, dtype=torch.int64, device=DEV),
                                        wl.scale, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert binding().device_status() == 0
    rows = np.union1d(sample_rows(wl, count=512).numpy(), glob)
    go, gl = gather_rows(out, lse, rows)
    del out, lse
    idx = torch.as_tensor(rows, device=DEV)
    ro, rl = oracle.attn_compressed(to_numpy_bits(q.index_select(0, idx)), to_numpy_bits(k),
                                    to_numpy_bits(v), wl.window, wl.block, glob, wl.scale,
                                    q_positions=rows)
    compare(go, ro, 1e-2, 1e-3, "compress 128K O (sampled + global rows)")
    compare(gl, rl, 1e-2, 1e-3, "compress 128K lse (sampled + global rows)")
