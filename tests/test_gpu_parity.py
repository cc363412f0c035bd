"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs -- landmark pooling, the fused window + landmark
attention (tensor-core kernel for bf16 / d=128, CUDA-core kernel otherwise),
Ring Attention partials and their LSE merge.  Small cases span several tiles
and ragged tails; the five workloads run in the launch configuration the
benchmark times, on all rows where the oracle finishes in seconds and on a
fixed row sample otherwise."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import (WORKLOADS, Workload, generate,
                                                          sample_rows, to_numpy_bits)
from tests.gpu_helpers import (bf16_round, bf16_ulp, binding, compare, gather_rows, gempty,
                               gempty_like, gfull, oracle_attention, run_gpu_attention, tol)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _oracle_threads():
    import os
    oracle.set_threads(os.cpu_count() or 1)


# ------------------------------------------------------------------ pooling
POOL_CASES = [(2048, 1, 64, 16, "f32"), (2048, 2, 128, 16, "bf16"), (32768, 1, 128, 512, "bf16"),
              (1000, 2, 64, 8, "f32"), (129, 1, 128, 129, "bf16"), (128, 3, 64, 1, "bf16"),
              pytest.param(131072, 8, 128, 512, "bf16", marks=pytest.mark.large)]


@pytest.mark.parametrize("n,Hkv,d,G,dt", POOL_CASES)
def test_landmark_pool_parity(n, Hkv, d, G, dt):
    B = binding()
    wl = Workload("pool", n, Hkv, Hkv, d, 1, G, dt, seed=n + G)
    _, k, v = generate(wl, device=DEV)
    k_lm = gempty((G, Hkv, d), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)
    torch.cuda.synchronize()
    for got, src in ((k_lm, k), (v_lm, v)):
        ref = oracle.landmark_pool(to_numpy_bits(src), G)
        g = got.float().cpu().numpy().astype(np.float64)
        if dt == "f32":
            compare(g, ref, 2e-6, 2e-7, f"pool f32 n={n}")
        else:
            # fp32 mean rounded to bf16: within one bf16 spacing of the exact mean
            assert np.all(np.abs(g - ref) <= bf16_ulp(bf16_round(ref))), f"pool bf16 n={n}"


# ------------------------------------------------------------------ attention, small grid
def _small_cases():
    heads = [(1, 1), (2, 1), (8, 1), (4, 2), (6, 6), (8, 2)]
    cases = []
    idx = 0
    for dt, d in (("bf16", 128), ("f32", 64), ("f32", 128), ("bf16", 64)):
        for n, G in ((1, 0), (1, 1), (127, 0), (127, 127), (128, 1), (128, 16), (129, 0),
                     (129, 3), (640, 5), (1000, 8), (1000, 1000)):
            B = n // G if G else n
            for w in sorted({1, max(1, B - 1), B, n, 300}):
                Hq, Hkv = heads[idx % len(heads)]
                idx += 1
                cases.append((dt, d, n, G, w, Hq, Hkv))
    return cases


@pytest.mark.parametrize("dt,d,n,G,w,Hq,Hkv", _small_cases())
def test_attention_small_grid(dt, d, n, G, w, Hq, Hkv):
    B = binding()
    wl = Workload("small", n, Hq, Hkv, d, w, G, dt, seed=7 * n + G + w)
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    ro, rl = oracle_attention(q, k, v, wl)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"O {wl}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"lse {wl}")
    assert B.uses_tensor_cores(Hq, Hkv, d, q.dtype) == (dt == "bf16" and d == 128)


def _random_cases(count=32, seed=20261203):
    """Seeded random shapes for both kernel families: ragged n, groups of one
    to eight query heads (odd ones leave a CTA of the pair idle in a slot),
    windows from one key to past n, landmark counts drawn from the divisors
    of n (or none); the work is capped so that the oracle finishes in
    seconds.  At the larger sizes a CTA pair takes several units in turn."""
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(count):
        dt, d = ("bf16", 128) if c % 4 else ("f32", 64)
        n = int(rng.integers(129, 5000))
        Hkv = int(rng.choice([1, 2, 3]))
        group = int(rng.choice([1, 2, 3, 4, 5, 8]))
        Hq = Hkv * group
        w = int(rng.integers(1, n + 100))
        w = max(1, min(w, int(4e7 // (n * Hq))))
        divisors = [g for g in range(1, n + 1) if n % g == 0]
        G = 0 if rng.random() < 0.2 else int(rng.choice(divisors))
        cases.append((dt, d, n, G, w, Hq, Hkv))
    return cases


@pytest.mark.parametrize("dt,d,n,G,w,Hq,Hkv", _random_cases())
def test_attention_random_shapes(dt, d, n, G, w, Hq, Hkv):
    wl = Workload("random", n, Hq, Hkv, d, w, G, dt, seed=n + 3 * w + G)
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    assert binding().device_status() == 0
    ro, rl = oracle_attention(q, k, v, wl)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"O {wl}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"lse {wl}")


def _random_ring_cases(count=8, seed=20261204):
    """Seeded ring rounds: uneven KV chunks (random cut points), a random
    order of the running merge, windows shorter or longer than a chunk."""
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(count):
        dt, d = ("bf16", 128) if c % 4 else ("f32", 64)
        n = int(rng.integers(300, 3000))
        Hkv = int(rng.choice([1, 2]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 6]))
        w = int(rng.integers(1, n + 1))
        chunks = int(rng.integers(2, 7))
        cuts = sorted(int(x) for x in rng.choice(np.arange(1, n), size=chunks - 1, replace=False))
        order = [int(x) for x in rng.permutation(chunks)]
        cases.append((dt, d, n, Hq, Hkv, w, tuple(cuts), tuple(order)))
    return cases


@pytest.mark.parametrize("dt,d,n,Hq,Hkv,w,cuts,order", _random_ring_cases())
def test_ring_random_chunks(dt, d, n, Hq, Hkv, w, cuts, order):
    """Each chunk's partial against the oracle restricted to that chunk
    (rows without a key: lse -inf, O untouched), and the rounds merged into
    a running result in a random order against the single pass."""
    B = binding()
    wl = Workload("ring_rand", n, Hq, Hkv, d, w, 0, dt, seed=n + w + len(cuts))
    q, k, v = generate(wl, device=DEV)
    bounds = [0, *cuts, n]
    pieces = [(bounds[i], bounds[i + 1]) for i in range(len(bounds) - 1)]
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    mx, mean = tol(dt)
    for lo, hi in pieces[:2]:
        o = gfull((n, Hq, d), 5.0, dtype=torch.float32, device=DEV)
        l = gempty((Hq, n), dtype=torch.float32, device=DEV)
        B.attn_fwd_partial(q, k[lo:hi], v[lo:hi], o, l, 0, lo, w, wl.scale)
        torch.cuda.synchronize()
        ro, rl = oracle.attn(qn, kn[lo:hi], vn[lo:hi], w, 0, wl.scale, kv_start=lo)
        compare(l.cpu().numpy(), rl, mx, mean, f"partial lse [{lo},{hi})")
        has = np.isfinite(rl[0])
        go = o.cpu().numpy()
        compare(go[has], ro[has], mx, mean, f"partial O [{lo},{hi})")
        assert np.all(go[~has] == 5.0), "rows without keys must be left untouched"
    out = gfull((n, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
    lse = gfull((Hq, n), -float("inf"), dtype=torch.float32, device=DEV)
    for i in order:
        lo, hi = pieces[i]
        B.attn_fwd_partial_merge(q, k[lo:hi], v[lo:hi], out, lse, 0, lo, w, wl.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    ro, rl = oracle.attn(qn, kn, vn, w, 0, wl.scale)
    compare(out.cpu().numpy(), ro, mx, mean, "running O")
    compare(lse.cpu().numpy(), rl, mx, mean, "running lse")


# ------------------------------------------------------------------ the five workloads
def test_pr1_2k_all_rows():
    wl = WORKLOADS["pr1_2k"]
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    ro, rl = oracle_attention(q, k, v, wl)
    compare(out.cpu().numpy(), ro, 1e-5, 1e-5, "pr1 O")
    compare(lse.cpu().numpy(), rl, 1e-5, 1e-5, "pr1 lse")


def test_32k_outliers_all_rows():
    wl = WORKLOADS["32k_outliers"]
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    ro, rl = oracle_attention(q, k, v, wl)
    compare(out.cpu().numpy(), ro, 1e-2, 1e-3, "32k O")
    compare(lse.cpu().numpy(), rl, 1e-2, 1e-3, "32k lse")


@pytest.mark.parametrize("name", ["128k_70b_layer", "1m_70b_layer"])
@pytest.mark.large
def test_large_workload_sampled_rows(name):
    wl = WORKLOADS[name]
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    rows = sample_rows(wl).numpy()
    go, gl = gather_rows(out, lse, rows)
    del out
    ro, rl = oracle_attention(q, k, v, wl, rows=rows)
    compare(go, ro, 1e-2, 1e-3, f"{name} O (sampled)")
    compare(gl, rl, 1e-2, 1e-3, f"{name} lse (sampled)")


@pytest.mark.large
def test_ring_128k_partials_and_merge():
    """8 KV chunks -> per-chunk partials -> LSE merge; equals the oracle's
    single-pass causal attention on sampled rows, and the GPU single pass
    on every row."""
    B = binding()
    wl = WORKLOADS["ring_128k"]
    q, k, v = generate(wl, device=DEV)
    n, Hq, d = q.shape
    c = n // wl.ring_chunks
    o_parts = [gempty((n, Hq, d), dtype=torch.float32, device=DEV)
               for _ in range(wl.ring_chunks)]
    l_parts = [gempty((Hq, n), dtype=torch.float32, device=DEV)
               for _ in range(wl.ring_chunks)]
    for p in range(wl.ring_chunks):
        B.attn_fwd_partial(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], o_parts[p], l_parts[p],
                           0, p * c, wl.window, wl.scale)
    merged = gempty((n, Hq, d), dtype=torch.float32, device=DEV)
    mlse = gempty((Hq, n), dtype=torch.float32, device=DEV)
    B.lse_merge(o_parts, l_parts, merged, mlse)
    # rows before a chunk have no key in it
    for p in range(1, wl.ring_chunks):
        assert bool(torch.isneginf(l_parts[p][:, : p * c]).all())
        assert bool(torch.isfinite(l_parts[p][:, p * c:]).all())
    del o_parts, l_parts
    single, slse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    compare(merged.cpu().numpy(), single.cpu().numpy(), 1e-2, 1e-3, "ring merged vs single")
    compare(mlse.cpu().numpy(), slse.cpu().numpy(), 1e-2, 1e-3, "ring lse merged vs single")
    rows = sample_rows(wl, count=512).numpy()
    go, gl = gather_rows(merged, mlse, rows)
    ro, rl = oracle_attention(q, k, v, wl, rows=rows)
    compare(go, ro, 1e-2, 1e-3, "ring merged O vs oracle")
    compare(gl, rl, 1e-2, 1e-3, "ring merged lse vs oracle")


# ------------------------------------------------------------------ partial + merge, small
@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
@pytest.mark.parametrize("n,chunks,w", [(512, 4, 512), (384, 3, 100), (1000, 8, 1000)])
def test_partial_merge_small(dt, d, n, chunks, w):
    B = binding()
    wl = Workload("ring_small", n, 4, 2, d, w, 0, dt, seed=n + chunks)
    q, k, v = generate(wl, device=DEV)
    bounds = np.linspace(0, n, chunks + 1).astype(int)
    o_parts, l_parts = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o = gfull((n, 4, d), 7.0, dtype=torch.float32, device=DEV)
        l = gempty((4, n), dtype=torch.float32, device=DEV)
        B.attn_fwd_partial(q, k[lo:hi], v[lo:hi], o, l, 0, int(lo), w, wl.scale)
        o_parts.append(o)
        l_parts.append(l)
    torch.cuda.synchronize()
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    mx, mean = tol(dt)
    for (lo, hi), o, l in zip(zip(bounds[:-1], bounds[1:]), o_parts, l_parts):
        ro, rl = oracle.attn(qn, kn[lo:hi], vn[lo:hi], w, 0, wl.scale, kv_start=int(lo))
        compare(l.cpu().numpy(), rl, mx, mean, f"partial lse [{lo},{hi})")
        has = np.isfinite(rl[0])
        go = o.cpu().numpy()
        compare(go[has], ro[has], mx, mean, f"partial O [{lo},{hi})")
        assert np.all(go[~has] == 7.0), "rows without keys must be left untouched"
    out = gempty((n, 4, d), dtype=torch.float32, device=DEV)
    lse = gempty((4, n), dtype=torch.float32, device=DEV)
    B.lse_merge(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.attn(qn, kn, vn, w, 0, wl.scale)
    compare(out.cpu().numpy(), ro, mx, mean, "merged O")
    compare(lse.cpu().numpy(), rl, mx, mean, "merged lse")


# ------------------------------------------------------------------ block band
@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
@pytest.mark.parametrize("n,bb,hw", [(1, 1, 0), (127, 128, 1), (128, 128, 0), (300, 128, 1),
                                     (1000, 128, 8), (1000, 64, 3), (513, 100, 2), (700, 128, 40)])
def test_band_small(dt, d, n, bb, hw):
    B = binding()
    wl = Workload("band_small", n, 8, 2, d, 1, 0, dt, seed=n + 17 * bb + hw)
    q, k, v = generate(wl, device=DEV)
    out = gempty((n, 8, d), dtype=torch.float32, device=DEV)
    lse = gempty((8, n), dtype=torch.float32, device=DEV)
    B.attn_fwd_band(q, k, v, out, lse, bb, hw, wl.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attn_band(to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v), bb, hw,
                              wl.scale)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"band O n={n} bb={bb} hw={hw}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"band lse n={n} bb={bb} hw={hw}")


def _random_band_cases(count=8, seed=20261206):
    """Seeded block bands: ragged n, block sizes that do and do not divide n
    or a 128-key tile, half-widths from zero blocks up, several groups."""
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(count):
        dt, d = ("bf16", 128) if c % 4 else ("f32", 64)
        n = int(rng.integers(100, 4000))
        Hkv = int(rng.choice([1, 2]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 5]))
        bb = int(rng.choice([1, 37, 64, 128, 200, 256]))
        hw = int(rng.integers(0, 6))
        cases.append((dt, d, n, Hq, Hkv, bb, hw))
    return cases


@pytest.mark.parametrize("dt,d,n,Hq,Hkv,bb,hw", _random_band_cases())
def test_band_random_shapes(dt, d, n, Hq, Hkv, bb, hw):
    B = binding()
    wl = Workload("band_rand", n, Hq, Hkv, d, 1, 0, dt, seed=n + bb + 5 * hw)
    q, k, v = generate(wl, device=DEV)
    out = gempty((n, Hq, d), dtype=torch.float32, device=DEV)
    lse = gempty((Hq, n), dtype=torch.float32, device=DEV)
    B.attn_fwd_band(q, k, v, out, lse, bb, hw, wl.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    ro, rl = oracle.attn_band(to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v), bb, hw,
                              wl.scale)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"band O {wl} bb={bb} hw={hw}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"band lse {wl} bb={bb} hw={hw}")


@pytest.mark.large
def test_band_128k_sampled_rows():
    import long_context_sparse_landmark_gb300.api as api
    wl = WORKLOADS["band_128k"]
    q, k, v = generate(wl, device=DEV)
    out, lse = api.band_attention(q, k, v, wl.band_block, wl.band_half, wl.scale,
                                  out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = sample_rows(wl).numpy()
    go, gl = gather_rows(out, lse, rows)
    idx = torch.as_tensor(rows, device=DEV)
    ro, rl = oracle.attn_band(to_numpy_bits(q.index_select(0, idx)), to_numpy_bits(k),
                              to_numpy_bits(v), wl.band_block, wl.band_half, wl.scale,
                              q_positions=rows)
    compare(go, ro, 1e-2, 1e-3, "band 128K O (sampled)")
    compare(gl, rl, 1e-2, 1e-3, "band 128K lse (sampled)")


# ------------------------------------------------------------------ fused ring rounds
@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64), ("bf16", 64), ("f32", 128)])
@pytest.mark.parametrize("n,chunks,w,order", [(512, 4, 512, "fwd"), (384, 3, 100, "rev"),
                                              (1000, 8, 1000, "mixed"), (257, 2, 64, "fwd")])
def test_partial_merge_running_result(dt, d, n, chunks, w, order):
    """Chunks merged into a running (O, lse) in any order equal the oracle's
    single pass; rows never reached keep their initial (garbage) O."""
    B = binding()
    wl = Workload("ring_run", n, 4, 2, d, w, 0, dt, seed=3 * n + chunks)
    q, k, v = generate(wl, device=DEV)
    bounds = np.linspace(0, n, chunks + 1).astype(int)
    pieces = list(zip(bounds[:-1], bounds[1:]))
    if order == "rev":
        pieces = pieces[::-1]
    elif order == "mixed":
        pieces = pieces[1::2] + pieces[0::2]
    out = gfull((n, 4, d), float("nan"), dtype=torch.float32, device=DEV)
    lse = gfull((4, n), -float("inf"), dtype=torch.float32, device=DEV)
    for lo, hi in pieces:
        B.attn_fwd_partial_merge(q, k[lo:hi], v[lo:hi], out, lse, 0, int(lo), w, wl.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attn(to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v), w, 0, wl.scale)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, "running O")
    compare(lse.cpu().numpy(), rl, mx, mean, "running lse")


@pytest.mark.large
def test_ring_128k_fused_rounds():
    """The ring workload through eight fused rounds equals the oracle on
    sampled rows and the separate partial + merge path on every row."""
    import long_context_sparse_landmark_gb300.api as api
    wl = WORKLOADS["ring_128k"]
    q, k, v = generate(wl, device=DEV)
    out, lse = api.ring_attention(q, k, v, wl.ring_chunks, fused=True)
    ref_o, ref_l = api.ring_attention(q, k, v, wl.ring_chunks, fused=False,
                                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    compare(out.cpu().numpy(), ref_o.cpu().numpy(), 1e-2, 1e-3, "fused vs separate O")
    compare(lse.cpu().numpy(), ref_l.cpu().numpy(), 1e-2, 1e-3, "fused vs separate lse")
    del ref_o
    rows = sample_rows(wl, count=512).numpy()
    go, gl = gather_rows(out, lse, rows)
    ro, rl = oracle_attention(q, k, v, wl, rows=rows)
    compare(go, ro, 1e-2, 1e-3, "fused ring O vs oracle")
    compare(gl, rl, 1e-2, 1e-3, "fused ring lse vs oracle")


# ------------------------------------------------------------------ merge alone
@pytest.mark.parametrize("P,n,Hq,d,out_dt", [(8, 1000, 4, 128, "f32"), (3, 257, 2, 64, "f32"),
                                             (64, 33, 2, 8, "f32"), (5, 500, 32, 128, "bf16"),
                                             (1, 17, 1, 4, "f32")])
def test_lse_merge_parity(P, n, Hq, d, out_dt):
    """Seeded random partials (some rows -inf in some parts, one row -inf in
    every part) merged on the GPU and by the oracle."""
    B = binding()
    g = torch.Generator(device="cpu").manual_seed(P * 1000 + n)
    o = torch.randn((P, n, Hq, d), generator=g, dtype=torch.float32)
    l = torch.randn((P, Hq, n), generator=g, dtype=torch.float32) * 3.0
    drop = torch.rand((P, Hq, n), generator=g) < 0.3
    l[drop] = -float("inf")
    l[:, :, 0] = -float("inf")
    o_d = [o[p].contiguous().to(DEV) for p in range(P)]
    l_d = [l[p].contiguous().to(DEV) for p in range(P)]
    tdt = torch.float32 if out_dt == "f32" else torch.bfloat16
    out = gempty((n, Hq, d), dtype=tdt, device=DEV)
    lse = gempty((Hq, n), dtype=torch.float32, device=DEV)
    B.lse_merge(o_d, l_d, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(o.double().numpy(), l.double().numpy())
    compare(lse.cpu().numpy(), rl, 2e-6, 2e-7, "merge lse")
    got = out.float().cpu().numpy()
    if out_dt == "f32":
        compare(got, ro, 1e-5, 1e-6, "merge O")
    else:
        assert np.all(np.abs(got - ro) <= bf16_ulp(bf16_round(ro)) + 1e-6)
    assert np.all(got[0] == 0.0)


def test_lse_merge_in_place():
    B = binding()
    g = torch.Generator(device="cpu").manual_seed(3)
    P, n, Hq, d = 4, 300, 8, 128
    o = torch.randn((P, n, Hq, d), generator=g)
    l = torch.randn((P, Hq, n), generator=g)
    o_d = [o[p].contiguous().to(DEV) for p in range(P)]
    l_d = [l[p].contiguous().to(DEV) for p in range(P)]
    B.lse_merge(o_d, l_d, o_d[0], l_d[0])
    torch.cuda.synchronize()
    ro, rl = oracle.lse_merge(o.double().numpy(), l.double().numpy())
    compare(o_d[0].cpu().numpy(), ro, 1e-5, 1e-6, "in-place merge O")
    compare(l_d[0].cpu().numpy(), rl, 2e-6, 2e-7, "in-place merge lse")


# ------------------------------------------------------------------ output dtype, determinism
def test_bf16_output_within_bars_plus_rounding():
    wl = Workload("bf16out", 2000, 8, 2, 128, 700, 8, "bf16", seed=11)
    q, k, v = generate(wl, device=DEV)
    out, lse = run_gpu_attention(q, k, v, wl, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ro, rl = oracle_attention(q, k, v, wl)
    got = out.float().cpu().numpy()
    # The bf16 output is the fp32 result rounded once: the fp32 bars apply
    # after allowing half a bf16 spacing for that rounding.
    excess = np.abs(got - ro) - 0.5 * bf16_ulp(ro)
    assert float(excess.max()) <= 1e-2, float(excess.max())
    assert float(np.abs(got - ro).mean()) <= 1e-3
    compare(lse.cpu().numpy(), rl, 1e-2, 1e-3, "lse")


@pytest.mark.large
def test_pair_kernel_128k_bf16_output_is_deterministic():
    """Three forward calls on the 128K layer with bf16 O (staged in shared
    memory, written by bulk tensor stores) give the same bits."""
    from long_context_sparse_landmark_gb300.workloads import WORKLOADS
    wl = WORKLOADS["128k_70b_layer"]
    q, k, v = generate(wl, device=DEV)
    o1, l1 = run_gpu_attention(q, k, v, wl, out_dtype=torch.bfloat16)
    for _ in range(2):
        o2, l2 = run_gpu_attention(q, k, v, wl, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        del o2, l2
    assert bool(torch.isfinite(o1.float()).all())
    assert binding().device_status() == 0


def test_tensor_core_kernel_is_deterministic():
    wl = Workload("det", 4096, 16, 2, 128, 1000, 16, "bf16", seed=5)
    q, k, v = generate(wl, device=DEV)
    o1, l1 = run_gpu_attention(q, k, v, wl)
    o2, l2 = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert binding().device_status() == 0
