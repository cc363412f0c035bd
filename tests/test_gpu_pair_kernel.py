"""The CTA-pair tensor-core attention kernel (two SMs share each MMA, used
for bf16, d = 128 with at least two query heads per KV head) against the
single-CTA tensor-core kernel, through the C ABI, bit for bit, in every mode
both serve: window + landmarks, row ranges, ring partials and running
merges, block band, selected blocks; fp32 and bf16 outputs.  Both kernels
compute the same per-row arithmetic in the same order, so their results
must be identical; each kernel is also checked against the fp64 oracle by
the parity tests (which run the pair kernel wherever it applies) and here
on the 128K layer's sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import (WORKLOADS, Workload, generate,
                                                          sample_rows, to_numpy_bits)
from tests.gpu_helpers import (binding, compare, gather_rows, gempty, gempty_like, gfull, gzeros,
                               oracle_attention, run_gpu_attention)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _oracle_threads():
    import os
    oracle.set_threads(os.cpu_count() or 1)


def both_kernels(run):
    """run() -> tuple of tensors, once with each kernel; returns (pair, single)."""
    B = binding()
    try:
        B.force_single_cta(False)
        a = [t.clone() for t in run()]
        torch.cuda.synchronize()
        assert B.device_status() == 0
        B.force_single_cta(True)
        b = [t.clone() for t in run()]
        torch.cuda.synchronize()
        assert B.device_status() == 0
    finally:
        B.force_single_cta(False)
    return a, b


def assert_same_bits(a, b, what):
    for x, y in zip(a, b):
        assert x.shape == y.shape
        same = torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x.view(torch.int16),
                           y.view(torch.int32) if y.dtype == torch.float32 else y.view(torch.int16))
        if not same:
            d = (x.float() - y.float()).abs()
            d = torch.where(torch.isnan(d), torch.zeros_like(d), d)
            raise AssertionError(f"{what}: kernels differ, max |diff| {float(d.max()):.3e}")


PLAIN_CASES = [
    # n, Hq, Hkv, w, G, out dtype
    (1, 2, 1, 1, 0, torch.float32),
    (127, 4, 2, 300, 127, torch.float32),
    (128, 2, 1, 64, 16, torch.bfloat16),
    (129, 6, 2, 129, 3, torch.float32),
    (640, 8, 1, 300, 5, torch.float32),
    (1000, 4, 1, 1, 8, torch.bfloat16),
    (1000, 6, 2, 125, 1000, torch.float32),
    (2048, 16, 2, 300, 16, torch.bfloat16),
    (4096, 8, 8 // 8, 1024, 32, torch.float32),
    (4096, 3 * 2, 2, 700, 64, torch.float32),   # group of 3: the last pair has one head
    (8192, 10, 2, 4096, 64, torch.bfloat16),    # group of 5
]


@pytest.mark.parametrize("n,Hq,Hkv,w,G,odt", PLAIN_CASES)
def test_pair_equals_single_window_landmarks(n, Hq, Hkv, w, G, odt):
    wl = Workload("pair", n, Hq, Hkv, 128, w, G, "bf16", seed=3 * n + Hq + G)
    q, k, v = generate(wl, device=DEV)
    a, b = both_kernels(lambda: run_gpu_attention(q, k, v, wl, out_dtype=odt))
    assert_same_bits(a, b, f"plain {wl} {odt}")


def test_pair_matches_oracle_small_groups():
    """Odd group sizes (idle second CTA on the last pair) against the oracle."""
    for n, Hq, Hkv, w, G in ((1000, 3, 1, 200, 8), (777, 10, 2, 300, 7)):
        wl = Workload("pair_o", n, Hq, Hkv, 128, w, G, "bf16", seed=n + Hq)
        q, k, v = generate(wl, device=DEV)
        out, lse = run_gpu_attention(q, k, v, wl)
        torch.cuda.synchronize()
        ro, rl = oracle_attention(q, k, v, wl)
        compare(out.cpu().numpy(), ro, 1e-2, 1e-3, f"pair O {wl}")
        compare(lse.cpu().numpy(), rl, 1e-2, 1e-3, f"pair lse {wl}")


def test_pair_equals_single_rows():
    """msa_attn_fwd_rows on ragged row ranges, lse with a row stride."""
    B = binding()
    wl = Workload("pair_rows", 3000, 8, 2, 128, 500, 12, "bf16", seed=41)
    q, k, v = generate(wl, device=DEV)
    k_lm = gempty((wl.G, wl.Hkv, 128), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)

    def run():
        out = gfull((wl.n, wl.Hq, 128), 7.0, device=DEV)
        lse = gfull((wl.Hq, wl.n), 7.0, device=DEV)
        for r0, r1 in ((0, 1), (1, 700), (700, 2048), (2048, 3000)):
            B.attn_fwd_rows(q[r0:r1], k, v, k_lm, v_lm, out[r0:r1], lse, r0, wl.window, wl.G,
                            wl.scale)
        return out, lse

    a, b = both_kernels(run)
    assert_same_bits(a, b, "rows")


def test_pair_equals_single_partials_and_merge():
    """Ring partials (rows without keys in a chunk get -inf) and the running
    merge, chunks in a scrambled order."""
    B = binding()
    wl = Workload("pair_ring", 4096, 8, 2, 128, 4096, 0, "bf16", seed=43)
    q, k, v = generate(wl, device=DEV)
    c = 1024

    def run_partials():
        outs = []
        for p_ in range(4):
            o = gfull((wl.n, wl.Hq, 128), 3.0, device=DEV)
            l_ = gempty((wl.Hq, wl.n), device=DEV)
            B.attn_fwd_partial(q, k[p_ * c:(p_ + 1) * c], v[p_ * c:(p_ + 1) * c], o, l_, 0, p_ * c,
                               wl.window, wl.scale)
            outs += [o, l_]
        return outs

    a, b = both_kernels(run_partials)
    assert_same_bits(a, b, "partials")

    def run_merge():
        o = gzeros((wl.n, wl.Hq, 128), device=DEV)
        l_ = gfull((wl.Hq, wl.n), float("-inf"), device=DEV)
        for p_ in (2, 0, 3, 1):
            B.attn_fwd_partial_merge(q, k[p_ * c:(p_ + 1) * c], v[p_ * c:(p_ + 1) * c], o, l_, 0,
                                     p_ * c, 1500, wl.scale)
        return o, l_

    a, b = both_kernels(run_merge)
    assert_same_bits(a, b, "running merge")


@pytest.mark.parametrize("n,bb,hw", [(1000, 128, 2), (4096, 128, 8), (2048, 64, 3)])
def test_pair_equals_single_band(n, bb, hw):
    B = binding()
    wl = Workload("pair_band", n, 8, 2, 128, 1, 0, "bf16", seed=n + bb)
    q, k, v = generate(wl, device=DEV)

    def run():
        out = gempty((n, 8, 128), device=DEV)
        lse = gempty((8, n), device=DEV)
        B.attn_fwd_band(q, k, v, out, lse, bb, hw, wl.scale)
        return out, lse

    a, b = both_kernels(run)
    assert_same_bits(a, b, f"band n={n}")


@pytest.mark.parametrize("n,G,w,top_k,Hq,Hkv", [(2048, 8, 300, 3, 8, 2), (8192, 16, 1000, 16, 16, 2),
                                                (4096, 32, 128, 6, 6, 2)])
def test_pair_equals_single_select(n, G, w, top_k, Hq, Hkv):
    B = binding()
    wl = Workload("pair_sel", n, Hq, Hkv, 128, w, G, "bf16", seed=n + G + top_k)
    q, k, v = generate(wl, device=DEV)
    k_lm = gempty((G, Hkv, 128), dtype=k.dtype, device=DEV)
    B.landmark_pool(k, v, k_lm, gempty_like(k_lm))
    n_qb = (n + 127) // 128
    sel = gempty((n_qb, Hkv, top_k), dtype=torch.int32, device=DEV)
    cnt = gempty((n_qb, Hkv), dtype=torch.int32, device=DEV)
    B.block_select(q, k_lm, sel, cnt, w, top_k)

    def run():
        out = gempty((n, Hq, 128), dtype=torch.bfloat16, device=DEV)
        lse = gempty((Hq, n), device=DEV)
        B.attn_fwd_select(q, k, v, sel, cnt, out, lse, w, G, top_k, wl.scale)
        return out, lse

    a, b = both_kernels(run)
    assert_same_bits(a, b, f"select {wl}")


@pytest.mark.large
def test_pair_128k_layer_sampled_rows_and_bits():
    """The 128K layer in the benchmark's launch configuration: the pair
    kernel's sampled rows against the oracle, and every row bit-equal to the
    single-CTA kernel."""
    wl = WORKLOADS["128k_70b_layer"]
    q, k, v = generate(wl, device=DEV)
    (out, lse), (out1, lse1) = both_kernels(lambda: run_gpu_attention(q, k, v, wl,
                                                                      out_dtype=torch.bfloat16))
    assert_same_bits((out, lse), (out1, lse1), "128K layer")
    del out1, lse1
    rows = sample_rows(wl, count=512).numpy()
    go, gl = gather_rows(out, lse, rows)
    ro, rl = oracle_attention(q, k, v, wl, rows=rows)
    # bf16 output: half a bf16 spacing on top of the fp32 bars (reading R10)
    err = np.abs(go - ro) - 0.5 * 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ro), 1e-30))) - 7)
    assert float(np.maximum(err, 0).max()) <= 1e-2
    compare(gl, rl, 1e-2, 1e-3, "128K lse (sampled)")


# ------------------------------------------------------------------ the persistent loop
def on_clusters(run, cap):
    """run() -> tuple of tensors, with the persistent pair kernels on at most
    `cap` CTA pairs (cap 0: as many as fit)."""
    B = binding()
    try:
        B.set_max_clusters(cap)
        r = [t.clone() for t in run()]
        torch.cuda.synchronize()
        assert B.device_status() == 0
    finally:
        B.set_max_clusters(0)
    return r


@pytest.mark.parametrize("cap", [1, 3])
def test_pair_kernels_on_few_clusters_equal_full_grid(cap):
    """On one or three CTA pairs every pair works through dozens of units in
    turn: barrier phases and tensor-memory slots carried from unit to unit,
    units of four heads next to units of one (a group of five), a slot idle
    on one CTA (a group of three), ring partials whose early query tiles
    have no key, a running merge, and the dQ kernel's units.  Each unit's
    arithmetic does not depend on which pair runs it, so every result equals
    the full grid's bit for bit."""
    B = binding()
    # window + landmarks, groups of five and of three
    for n, Hq, Hkv, w, G, odt in ((2048, 10, 2, 1024, 16, torch.bfloat16),
                                  (4096, 6, 2, 700, 64, torch.float32)):
        wl = Workload("pair_cap", n, Hq, Hkv, 128, w, G, "bf16", seed=5 * n + Hq)
        q, k, v = generate(wl, device=DEV)

        def run_plain():
            return run_gpu_attention(q, k, v, wl, out_dtype=odt)

        assert_same_bits(on_clusters(run_plain, cap), on_clusters(run_plain, 0),
                         f"plain {wl} on {cap} pairs")

    # ring partials (T = 0 units) and a running merge
    wl = Workload("pair_cap_ring", 2048, 8, 2, 128, 2048, 0, "bf16", seed=47)
    q, k, v = generate(wl, device=DEV)
    c = 512

    def run_ring():
        outs = []
        for p_ in (3, 1):
            o = gfull((wl.n, wl.Hq, 128), 3.0, device=DEV)
            l_ = gempty((wl.Hq, wl.n), device=DEV)
            B.attn_fwd_partial(q, k[p_ * c:(p_ + 1) * c], v[p_ * c:(p_ + 1) * c], o, l_, 0, p_ * c,
                               wl.window, wl.scale)
            outs += [o, l_]
        o = gzeros((wl.n, wl.Hq, 128), device=DEV)
        l_ = gfull((wl.Hq, wl.n), float("-inf"), device=DEV)
        for p_ in (2, 0, 3, 1):
            B.attn_fwd_partial_merge(q, k[p_ * c:(p_ + 1) * c], v[p_ * c:(p_ + 1) * c], o, l_, 0,
                                     p_ * c, 700, wl.scale)
        return outs + [o, l_]

    assert_same_bits(on_clusters(run_ring, cap), on_clusters(run_ring, 0),
                     f"ring partials and merge on {cap} pairs")

    # the dQ pair kernel (an even group): 16 query tiles x 2 head pairs x 2 KV heads
    wl = Workload("pair_cap_bwd", 2048, 8, 2, 128, 600, 16, "bf16", seed=53)
    q, k, v = generate(wl, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(59)
    do = torch.randn((wl.n, wl.Hq, 128), generator=gen, device=DEV).to(torch.bfloat16)
    k_lm = gempty((wl.G, wl.Hkv, 128), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)
    out = gempty((wl.n, wl.Hq, 128), device=DEV)
    lse = gempty((wl.Hq, wl.n), device=DEV)
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale)
    ws = gempty((B.attn_bwd_workspace_size(wl.n, wl.Hq, wl.Hkv, 128, wl.G),), dtype=torch.uint8,
                device=DEV)

    def run_bwd():
        dq = gempty((wl.n, wl.Hq, 128), device=DEV)
        dk = gempty((wl.n, wl.Hkv, 128), device=DEV)
        dv = gempty_like(dk)
        B.attn_bwd(q, k, v, k_lm, v_lm, out, lse, do, dq, dk, dv, wl.window, wl.G, wl.scale, ws)
        return dq, dk, dv

    assert_same_bits(on_clusters(run_bwd, cap), on_clusters(run_bwd, 0), f"backward on {cap} pairs")
