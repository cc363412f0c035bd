"""GPU parity of landmark-scored top-k block selection and of attention over
window + selected blocks, through the C ABI, against the fp64 oracle.

Selection is an integer decision taken from floating-point scores: the GPU
scores with bf16 (or fp32) block-mean keys and fp32 sums, the oracle in
fp64.  Counts must match exactly.  Where the oracle's k-th and (k+1)-th
scores are further apart than the GPU's worst-case scoring error the chosen
set is unique and must match exactly; otherwise any set the GPU's rounding
could have produced is accepted (every chosen block's exact score, plus the
error bound, reaches every unchosen candidate's, minus it).  Attention is
checked with the oracle's own selection fed to the GPU, and the fused
pool -> select -> attend call on every (row, head) pair: where the GPU's
selection is the oracle's against the oracle end to end, and everywhere
against the oracle's attention over the GPU's own selection, once that
selection has been checked to be one the scores allow."""
import math

import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import (WORKLOADS, Workload, generate,
                                                          sample_rows, to_numpy_bits)
from tests.gpu_helpers import binding, compare, gather_rows, gempty, gempty_like, gfull, tol

pytestmark = pytest.mark.gpu

DEV = "cuda"
QB = 128  # query rows per selection block


@pytest.fixture(scope="module", autouse=True)
def _oracle_threads():
    import os
    oracle.set_threads(os.cpu_count() or 1)


def gpu_select(q, k, v, G, window, top_k):
    """Pool K (msa_landmark_pool) and select (msa_block_select) on the GPU."""
    B = binding()
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    k_lm = gempty((G, Hkv, d), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)
    n_qb = (n + QB - 1) // QB
    sel = gfull((n_qb, Hkv, top_k), -7, dtype=torch.int32, device=DEV)
    cnt = gfull((n_qb, Hkv), -7, dtype=torch.int32, device=DEV)
    B.block_select(q, k_lm, sel, cnt, window, top_k)
    return sel, cnt


def score_error_bound(q, k, G):
    """Per (query block, KV group, key block) bound on |GPU score - exact|:
    bf16 rounding of the block-mean key (relative 2^-9, taken as 2^-8) on
    the exact query sum, plus fp32 summation of the queries and of the dot
    product (taken as 2^-12 of the absolute sums)."""
    qf = q.double().cpu().numpy()
    n, Hq, d = qf.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    n_qb = (n + QB - 1) // QB
    pad = np.zeros((n_qb * QB, Hq, d))
    pad[:n] = qf
    qa = pad.reshape(n_qb, QB, Hkv, g, d)
    qsum = np.abs(qa.sum(axis=(1, 3)))
    qabs = np.abs(qa).sum(axis=(1, 3))
    kab = np.abs(oracle.landmark_pool(to_numpy_bits(k), G))
    return (2.0 ** -8 * np.einsum("tcd,gcd->tcg", qsum, kab)
            + 2.0 ** -12 * np.einsum("tcd,gcd->tcg", qabs, kab))


def check_selection(sel_g, cnt_g, scores, eps, top_k):
    """Returns the [n_qb, Hkv] mask of units whose GPU set equals the
    oracle's; asserts validity everywhere."""
    sel_o, cnt_o = oracle.select_top_k(scores, top_k)
    assert np.array_equal(cnt_g, cnt_o), "selection counts differ"
    used = np.arange(top_k)[None, None, :] < cnt_o[:, :, None]
    same = ((sel_g == sel_o) | ~used).all(axis=2)
    for t, c in zip(*np.nonzero(~same)):
        k_ = int(cnt_o[t, c])
        chosen = sel_g[t, c, :k_]
        assert np.all(np.diff(chosen) > 0), f"unit ({t},{c}): not ascending/distinct"
        assert np.all((chosen >= 0) & (chosen < scores.shape[2]))
        s, e = scores[t, c], eps[t, c]
        assert np.all(np.isfinite(s[chosen])), f"unit ({t},{c}): chose a non-candidate"
        cand = np.nonzero(np.isfinite(s))[0]
        unchosen = np.setdiff1d(cand, chosen)
        if unchosen.size:
            lo = float((s[chosen] + e[chosen]).min())
            hi = float((s[unchosen] - e[unchosen]).max())
            assert lo >= hi, f"unit ({t},{c}): chosen {lo:.4g} below unchosen {hi:.4g}"
    return same


SELECT_CASES = [
    # dt, d, n, G, w, top_k, Hq, Hkv
    ("bf16", 128, 2048, 8, 300, 3, 8, 2),
    ("bf16", 128, 1000, 8, 100, 2, 4, 1),
    ("f32", 64, 1000, 8, 100, 2, 4, 1),
    ("bf16", 64, 2048, 16, 128, 16, 6, 6),
    ("f32", 128, 128, 128, 1, 128, 2, 1),
    ("bf16", 128, 1024, 1, 1, 1, 2, 2),
    ("bf16", 128, 4096, 1024, 64, 40, 8, 1),
    ("bf16", 128, 16384, 64, 1024, 8, 16, 2),
    ("f32", 128, 777, 7, 1, 7, 3, 3),
]


@pytest.mark.parametrize("dt,d,n,G,w,top_k,Hq,Hkv", SELECT_CASES)
def test_block_select_valid(dt, d, n, G, w, top_k, Hq, Hkv):
    wl = Workload("sel", n, Hq, Hkv, d, w, G, dt, seed=3 * n + G + top_k)
    q, k, v = generate(wl, device=DEV)
    sel, cnt = gpu_select(q, k, v, G, w, top_k)
    torch.cuda.synchronize()
    scores = oracle.block_scores(to_numpy_bits(q), to_numpy_bits(k), G, w)
    eps = score_error_bound(q, k, G)
    same = check_selection(sel.cpu().numpy(), cnt.cpu().numpy(), scores, eps, top_k)
    if dt == "f32":
        assert same.all(), "fp32 selection differs from the oracle"
    assert binding().device_status() == 0


def test_block_select_ties_to_lower_index():
    """K = 0 (every score 0) and K built from one repeated block (equal
    landmarks): the lowest-index candidates win, exactly as the oracle."""
    n, Hq, Hkv, d, G, w, top_k = 4096, 8, 2, 128, 32, 200, 5
    wl = Workload("ties", n, Hq, Hkv, d, w, G, "bf16", seed=11)
    q, k, v = generate(wl, device=DEV)
    B = n // G
    for kk in (torch.zeros_like(k), k[:B].repeat(G, 1, 1).contiguous()):
        sel, cnt = gpu_select(q, kk, v, G, w, top_k)
        torch.cuda.synchronize()
        scores = oracle.block_scores(to_numpy_bits(q), to_numpy_bits(kk), G, w)
        sel_o, cnt_o = oracle.select_top_k(scores, top_k)
        assert np.array_equal(cnt.cpu().numpy(), cnt_o)
        used = np.arange(top_k)[None, None, :] < cnt_o[:, :, None]
        assert np.array_equal(np.where(used, sel.cpu().numpy(), 0), np.where(used, sel_o, 0))


def test_block_select_planted_block():
    """Queries share a direction u; block 3's keys are shifted along u, so it
    outscores every other block wherever it is a candidate (top-1)."""
    n, Hq, Hkv, d, G, w = 4096, 8, 2, 128, 16, 512
    wl = Workload("plant", n, Hq, Hkv, d, w, G, "bf16", seed=5)
    q, k, v = generate(wl, device=DEV)
    u = torch.ones(d, device=DEV) / math.sqrt(d)
    q = (q.float() + u).to(torch.bfloat16)
    Bk = n // G
    k = k.float()
    k[3 * Bk:4 * Bk] += 4.0 * u
    k = k.to(torch.bfloat16)
    sel, cnt = gpu_select(q, k, v, G, w, 1)
    torch.cuda.synchronize()
    sel = sel.cpu().numpy()
    t_first = next(t for t in range(n // QB) if (3 + 1) * Bk <= t * QB - w + 1)
    assert (sel[t_first:, :, 0] == 3).all()
    scores = oracle.block_scores(to_numpy_bits(q), to_numpy_bits(k), G, w)
    sel_o, _ = oracle.select_top_k(scores, 1)
    assert (sel_o[t_first:, :, 0] == 3).all()


ATTN_CASES = [
    # dt, d, n, G, w, top_k, Hq, Hkv   (tensor-core path: bf16, d=128, block % 128 == 0)
    ("bf16", 128, 2048, 8, 300, 3, 8, 2),
    ("bf16", 128, 4096, 32, 128, 6, 4, 1),
    ("bf16", 128, 1024, 1, 1, 1, 2, 2),
    ("bf16", 128, 8192, 16, 1000, 16, 16, 2),
    ("bf16", 128, 1000, 8, 100, 2, 4, 1),
    ("f32", 64, 1000, 8, 100, 2, 4, 1),
    ("bf16", 64, 2048, 16, 128, 16, 6, 6),
    ("f32", 128, 128, 128, 1, 128, 2, 1),
    ("f32", 128, 777, 7, 1, 7, 3, 3),
]


@pytest.mark.parametrize("dt,d,n,G,w,top_k,Hq,Hkv", ATTN_CASES)
def test_attn_select_oracle_selection(dt, d, n, G, w, top_k, Hq, Hkv):
    """msa_attn_fwd_select given the oracle's selection equals the oracle."""
    B = binding()
    wl = Workload("asel", n, Hq, Hkv, d, w, G, dt, seed=5 * n + G + w)
    q, k, v = generate(wl, device=DEV)
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    sel_o, cnt_o = oracle.select_top_k(oracle.block_scores(qn, kn, G, w), top_k)
    sel = torch.from_numpy(np.ascontiguousarray(sel_o)).to(DEV)
    cnt = torch.from_numpy(np.ascontiguousarray(cnt_o)).to(DEV)
    out = gempty((n, Hq, d), dtype=torch.float32, device=DEV)
    lse = gempty((Hq, n), dtype=torch.float32, device=DEV)
    B.attn_fwd_select(q, k, v, sel, cnt, out, lse, w, G, top_k, wl.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    ro, rl = oracle.attn_select(qn, kn, vn, w, G, sel_o, cnt_o, wl.scale)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, f"select O {wl}")
    compare(lse.cpu().numpy(), rl, mx, mean, f"select lse {wl}")
    assert B.uses_tensor_cores(Hq, Hkv, d, q.dtype) == (dt == "bf16" and d == 128)


def _fused_vs_steps(q, k, v, wl):
    """The one-call path equals pool -> select -> attend run step by step,
    bit for bit; returns the steps' selection and output."""
    B = binding()
    import long_context_sparse_landmark_gb300.api as api
    out_f, lse_f = api.topk_attention(q, k, v, wl.window, wl.G, wl.top_k, wl.scale,
                                      out_dtype=torch.float32)
    sel, cnt = gpu_select(q, k, v, wl.G, wl.window, wl.top_k)
    out = gempty_like(out_f)
    lse = gempty_like(lse_f)
    B.attn_fwd_select(q, k, v, sel, cnt, out, lse, wl.window, wl.G, wl.top_k, wl.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert torch.equal(out_f, out) and torch.equal(lse_f, lse), "fused != step by step"
    del out_f, lse_f
    return sel.cpu().numpy(), cnt.cpu().numpy(), out, lse


@pytest.mark.parametrize("dt,d,n,G,w,top_k,Hq,Hkv", ATTN_CASES[:7])
def test_topk_fused_against_oracle(dt, d, n, G, w, top_k, Hq, Hkv):
    wl = Workload("fused", n, Hq, Hkv, d, w, G, dt, seed=n + 13 * G, top_k=top_k)
    q, k, v = generate(wl, device=DEV)
    sel, cnt, out, lse = _fused_vs_steps(q, k, v, wl)
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    scores = oracle.block_scores(qn, kn, G, w)
    same = check_selection(sel, cnt, scores, score_error_bound(q, k, G), top_k)
    sel_o, cnt_o = oracle.select_top_k(scores, top_k)
    ro, rl = oracle.attn_select(qn, kn, vn, w, G, sel_o, cnt_o, wl.scale)
    # (row, head) pairs whose KV group chose the oracle's set: end to end
    g = Hq // Hkv
    keep = np.repeat(same, g, axis=1)[np.arange(n) // QB]          # [n, Hq]
    assert keep.mean() > 0.5, f"only {keep.mean():.2f} of (row, head) pairs comparable"
    mx, mean = tol(dt)
    o = out.cpu().numpy()
    l_ = lse.cpu().numpy()
    compare(o[keep], ro[keep], mx, mean, f"fused O {wl}")
    compare(l_[keep.T], rl[keep.T], mx, mean, f"fused lse {wl}")
    # every pair: the oracle's attention over the GPU's (validated) selection
    rg, rgl = oracle.attn_select(qn, kn, vn, w, G, sel, cnt, wl.scale)
    compare(o, rg, mx, mean, f"fused O, GPU selection {wl}")
    compare(l_, rgl, mx, mean, f"fused lse, GPU selection {wl}")


def _random_topk_cases(count=8, seed=20261207):
    """Seeded top-k shapes: key blocks of whole 128-key tiles (tensor-core
    path) or not (fp32 / d = 64 on the CUDA-core kernel), top_k from one to
    every block, windows shorter and longer than a block, several groups."""
    rng = np.random.default_rng(seed)
    cases = []
    for c in range(count):
        Hkv = int(rng.choice([1, 2]))
        Hq = Hkv * int(rng.choice([1, 2, 3, 4]))
        if c % 4:
            dt, d = "bf16", 128
            block = 128 * int(rng.integers(1, 4))
        else:
            dt, d = "f32", 64
            block = int(rng.integers(20, 300))
        G = int(rng.integers(2, 24))
        n = G * block
        w = int(rng.integers(1, 3 * block))
        top_k = int(rng.integers(1, G + 1))
        cases.append((dt, d, n, G, w, top_k, Hq, Hkv))
    return cases


@pytest.mark.parametrize("dt,d,n,G,w,top_k,Hq,Hkv", _random_topk_cases())
def test_topk_random_shapes(dt, d, n, G, w, top_k, Hq, Hkv):
    """The one-call path equals the three steps bit for bit; its selection
    is valid against the oracle's scores; its output equals the oracle's
    attention over that selection, and over the oracle's own selection in
    the KV groups where the two agree."""
    wl = Workload("topk_rand", n, Hq, Hkv, d, w, G, dt, seed=n + 7 * w + top_k, top_k=top_k)
    q, k, v = generate(wl, device=DEV)
    sel, cnt, out, lse = _fused_vs_steps(q, k, v, wl)
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    scores = oracle.block_scores(qn, kn, G, w)
    same = check_selection(sel, cnt, scores, score_error_bound(q, k, G), top_k)
    mx, mean = tol(dt)
    o = out.cpu().numpy()
    l_ = lse.cpu().numpy()
    rg, rgl = oracle.attn_select(qn, kn, vn, w, G, sel, cnt, wl.scale)
    compare(o, rg, mx, mean, f"top-k O, GPU selection {wl}")
    compare(l_, rgl, mx, mean, f"top-k lse, GPU selection {wl}")
    sel_o, cnt_o = oracle.select_top_k(scores, top_k)
    ro, rl = oracle.attn_select(qn, kn, vn, w, G, sel_o, cnt_o, wl.scale)
    keep = np.repeat(same, Hq // Hkv, axis=1)[np.arange(n) // QB]      # [n, Hq]
    if keep.any():
        compare(o[keep], ro[keep], mx, mean, f"top-k O, oracle selection {wl}")
        compare(l_[keep.T], rl[keep.T], mx, mean, f"top-k lse, oracle selection {wl}")


@pytest.mark.large
def test_topk_128k_sampled_rows():
    """The 128K top-k workload in the benchmark's launch configuration:
    fused call == steps, selection valid on every unit, sampled rows equal
    the oracle where the selection is the oracle's, and every sampled row
    and head equal to the oracle's attention over the GPU's selection."""
    wl = WORKLOADS["topk_128k"]
    q, k, v = generate(wl, device=DEV)
    sel, cnt, out, lse = _fused_vs_steps(q, k, v, wl)
    qn, kn, vn = to_numpy_bits(q), to_numpy_bits(k), to_numpy_bits(v)
    scores = oracle.block_scores(qn, kn, wl.G, wl.window)
    same = check_selection(sel, cnt, scores, score_error_bound(q, k, wl.G), wl.top_k)
    assert same.mean() > 0.5, f"only {same.mean():.2f} of units match the oracle's set"
    sel_o, cnt_o = oracle.select_top_k(scores, wl.top_k)
    rows = sample_rows(wl, count=512).numpy()
    go, gl = gather_rows(out, lse, rows)
    del out, lse
    idx = torch.as_tensor(rows, device=DEV)
    ro, rl = oracle.attn_select(to_numpy_bits(q.index_select(0, idx)), kn, vn, wl.window, wl.G,
                                sel_o, cnt_o, wl.scale, q_positions=rows)
    keep = np.repeat(same, wl.Hq // wl.Hkv, axis=1)[rows // QB]      # [rows, Hq]
    compare(go[keep], ro[keep], 1e-2, 1e-3, "topk 128K O (sampled)")
    compare(gl[keep.T], rl[keep.T], 1e-2, 1e-3, "topk 128K lse (sampled)")
    # every sampled row and head, units whose selection differs included
    rg, rgl = oracle.attn_select(to_numpy_bits(q.index_select(0, idx)), kn, vn, wl.window, wl.G,
                                 sel, cnt, wl.scale, q_positions=rows)
    compare(go, rg, 1e-2, 1e-3, "topk 128K O, GPU selection (sampled)")
    compare(gl, rgl, 1e-2, 1e-3, "topk 128K lse, GPU selection (sampled)")
    print(f"128K top-k: {100 * (1 - same.mean()):.1f}% of units chose a set other than the "
          "oracle's (each checked valid and compared through the oracle)")


def test_attn_select_rejects_bad_selection_without_reading_out_of_bounds():
    """A count above top_k and block indices that are not candidates are
    clamped by the kernels and reported as MSA_ERR_INVALID_ARG."""
    B = binding()
    n, Hq, Hkv, d, G, w, top_k = 2048, 4, 1, 128, 8, 256, 2
    for dt in ("bf16", "f32"):
        wl = Workload("bad", n, Hq, Hkv, d, w, G, dt, seed=1)
        q, k, v = generate(wl, device=DEV)
        n_qb = n // QB
        sel = gfull((n_qb, Hkv, top_k), 10 ** 6, dtype=torch.int32, device=DEV)
        cnt = gfull((n_qb, Hkv), 99, dtype=torch.int32, device=DEV)
        out = gempty((n, Hq, d), dtype=torch.float32, device=DEV)
        lse = gempty((Hq, n), dtype=torch.float32, device=DEV)
        B.device_status(clear=True)
        B.attn_fwd_select(q, k, v, sel, cnt, out, lse, w, G, top_k, wl.scale)
        torch.cuda.synchronize()
        assert B.device_status(clear=True) == 1  # MSA_ERR_INVALID_ARG
        assert torch.isfinite(out).all()
