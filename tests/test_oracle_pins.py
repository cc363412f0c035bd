"""Pins for the fp64 CPU oracle (no GPU).

The oracle is only trusted because these checks tie it to something other
than itself: a dense brute force written from the set definitions, exact
causal attention from a library routine, the merge invariant of Ring
Attention ("Training at 1M+ Token Context", Ring Attention paragraph: each
round aggregates softmax statistics), convexity, closed forms, and the
page's own dot-product counts ("Scaling GPU Cluster for Million Token
Context", section "The Cost of Attention: O(n^2) vs Sparse").
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from long_context_sparse_landmark_gb300.workloads import WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- brute force
def dense_bruteforce(q, k, v, window, G, scale):
    """Materialise the full [n, n+G] masked score matrix per head (numpy).

    Independent of the oracle: the mask is built element by element from the
    two set definitions (window i-w < j <= i; landmark l visible when its
    whole block [lB, (l+1)B) ends at or before i-w+1), landmarks come from
    numpy's block mean, the softmax is taken over the masked row.
    """
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    if G > 0:
        B = n // G
        klm = k.reshape(G, B, Hkv, d).mean(axis=1)
        vlm = v.reshape(G, B, Hkv, d).mean(axis=1)
    else:
        B = 1
        klm = np.zeros((0, Hkv, d))
        vlm = np.zeros((0, Hkv, d))
    mask = np.zeros((n, n + G), dtype=bool)
    for i in range(n):
        for j in range(n):
            mask[i, j] = (i - window < j) and (j <= i)
        for l in range(G):
            block_last = (l + 1) * B - 1
            mask[i, n + l] = block_last <= i - window
    out = np.zeros((n, Hq, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        c = h // g
        keys = np.concatenate([k[:, c], klm[:, c]], axis=0)
        vals = np.concatenate([v[:, c], vlm[:, c]], axis=0)
        s = scale * q[:, h] @ keys.T
        s = np.where(mask, s, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        e = np.where(mask, np.exp(s - mx), 0.0)
        den = e.sum(axis=1, keepdims=True)
        out[:, h] = (e / den) @ vals
        lse[h] = (mx + np.log(den))[:, 0]
    return out, lse


def to_bits(x32):
    """fp32 array -> bf16 bit patterns (round to nearest even) and the fp32
    values those bits hold."""
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.to(torch.float32).numpy()


def rand_qkv(rng, n, Hq, Hkv, d):
    q = rng.standard_normal((n, Hq, d)).astype(np.float32)
    k = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    v = rng.standard_normal((n, Hkv, d)).astype(np.float32)
    return q, k, v


def landmark_count(i, window, G, B):
    """L(i) = clamp(floor((i - w + 1) / B), 0, G), the closed form."""
    if G == 0:
        return 0
    return int(min(G, max(0, (i - window + 1) // B)))


# ------------------------------------------------------------------- P1
CASES = []
for (n, G) in [(1, 0), (1, 1), (7, 0), (7, 7), (16, 0), (16, 1), (16, 2),
               (16, 4), (16, 8), (16, 16), (48, 6), (64, 8)]:
    B = n // G if G else 1
    for w in sorted({1, 2, max(1, B - 1), B, B + 1, n, n + 5}):
        CASES.append((n, G, w))


@pytest.mark.parametrize("n,G,w", CASES)
def test_p1_bruteforce(oracle_mod, n, G, w):
    rng = np.random.default_rng(1000 * n + 10 * G + w)
    for (Hq, Hkv), d in itertools.product([(1, 1), (2, 1), (4, 2), (4, 1)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        scale = 1.0 / math.sqrt(d)
        ref_o, ref_l = dense_bruteforce(q, k, v, w, G, scale)
        o, l = oracle_mod.attn(q, k, v, w, G, scale)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_p1_bruteforce_bf16_storage(oracle_mod):
    """bf16 bit patterns are read as the values they encode."""
    rng = np.random.default_rng(7)
    n, G, w, Hq, Hkv, d = 32, 4, 5, 4, 2, 8
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    (qb, qf), (kb, kf), (vb, vf) = to_bits(q), to_bits(k), to_bits(v)
    ref_o, ref_l = dense_bruteforce(qf, kf, vf, w, G, 0.3)
    o, l = oracle_mod.attn(qb, kb, vb, w, G, 0.3)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_p1_sampled_rows_match_all_rows(oracle_mod):
    rng = np.random.default_rng(3)
    q, k, v = rand_qkv(rng, 64, 4, 2, 8)
    o, l = oracle_mod.attn(q, k, v, 9, 8, 0.35)
    rows = np.array([0, 5, 17, 63])
    os_, ls_ = oracle_mod.attn(q, k, v, 9, 8, 0.35, rows=rows)
    np.testing.assert_array_equal(os_, o[rows])
    np.testing.assert_array_equal(ls_, l[:, rows])


# ------------------------------------------------------------------- P2
@pytest.mark.parametrize("n,Hq,Hkv,d", [(1, 1, 1, 4), (33, 4, 2, 8),
                                        (128, 8, 1, 16), (200, 4, 4, 32)])
def test_p2_causal_special_case(oracle_mod, n, Hq, Hkv, d):
    """w >= n and G = 0 is exact causal attention (torch SDPA, fp64, CPU)."""
    rng = np.random.default_rng(n)
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    for w in (n, n + 17):
        o, _ = oracle_mod.attn(q, k, v, w, 0, scale)
        g = Hq // Hkv
        tq = torch.from_numpy(q).double().permute(1, 0, 2)[None]
        tk = torch.from_numpy(k).double().repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
        tv = torch.from_numpy(v).double().repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, is_causal=True, scale=scale)[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------- P3
def _chunked(oracle_mod, q, k, v, w, scale, bounds):
    parts_o, parts_l = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o, l = oracle_mod.attn(q, k[lo:hi], v[lo:hi], w, 0, scale, kv_start=lo)
        parts_o.append(o)
        parts_l.append(l)
    return np.stack(parts_o), np.stack(parts_l)


@pytest.mark.parametrize("w", [1, 5, 40, 1000])
def test_p3_merge_of_chunks_equals_single_pass(oracle_mod, w):
    rng = np.random.default_rng(w)
    n, Hq, Hkv, d = 96, 4, 2, 8
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    scale = 0.4
    ref_o, ref_l = oracle_mod.attn(q, k, v, w, 0, scale)
    for bounds in ([0, 1, 8, 96], [0, 7, 14, 21, 28, 35, 42, 49, 56, 63, 70, 77, 84, 91, 96],
                   [0, 12, 24, 36, 48, 60, 72, 84, 96], [0, 50, 51, 96], [0, 96]):
        po, pl = _chunked(oracle_mod, q, k, v, w, scale, bounds)
        o, l = oracle_mod.lse_merge(po, pl)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_p3_merge_pr1_size(oracle_mod):
    """Causal attention on the 2048-token fp32 shape: 8 chunks merged."""
    wl = WORKLOADS["pr1_2k"]
    rng = np.random.default_rng(0)
    q, k, v = rand_qkv(rng, wl.n, wl.Hq, wl.Hkv, wl.d)
    rows = np.arange(0, wl.n, 7)
    ref_o, ref_l = oracle_mod.attn(q, k, v, wl.n, 0, wl.scale, rows=rows)
    bounds = list(range(0, wl.n + 1, wl.n // 8))
    parts_o, parts_l = [], []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        o, l = oracle_mod.attn(q, k[lo:hi], v[lo:hi], wl.n, 0, wl.scale,
                               rows=rows, kv_start=lo)
        parts_o.append(o)
        parts_l.append(l)
    o, l = oracle_mod.lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_p3_empty_parts(oracle_mod):
    """A chunk entirely after a row gives lse = -inf and is skipped."""
    rng = np.random.default_rng(5)
    q, k, v = rand_qkv(rng, 16, 2, 1, 4)
    o, l = oracle_mod.attn(q, k[8:], v[8:], 16, 0, 0.5, kv_start=8)
    assert np.all(np.isneginf(l[:, :8]))
    assert np.all(o[:8] == 0.0)
    assert np.all(np.isfinite(l[:, 8:]))
    mo, ml = oracle_mod.lse_merge(np.stack([o, o]), np.stack([l, l]))
    assert np.all(np.isneginf(ml[:, :8]))
    np.testing.assert_allclose(mo[8:], o[8:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml[:, 8:], l[:, 8:] + math.log(2.0), rtol=0, atol=1e-12)


# ------------------------------------------------------------------- P4
@pytest.mark.parametrize("n,G,w", [(16, 4, 3), (24, 6, 1), (32, 8, 9), (12, 12, 2)])
def test_p4_weights_are_a_convex_combination(oracle_mod, n, G, w):
    """With V = identity (d = n), O[i, k] is the weight the row puts on
    token k (window part plus its block's landmark share / B): all weights
    are >= 0 and they sum to 1."""
    rng = np.random.default_rng(n + G)
    d = n
    q = rng.standard_normal((n, 2, d)).astype(np.float32)
    k = rng.standard_normal((n, 1, d)).astype(np.float32)
    v = np.eye(n, dtype=np.float32)[:, None, :]
    o, _ = oracle_mod.attn(q, k, v, w, G, 0.3)
    assert np.all(o >= -1e-15)
    np.testing.assert_allclose(o.sum(axis=2), 1.0, rtol=0, atol=1e-12)
    # Weight sits only on attended tokens: the window, or a visible block.
    B = n // G
    for i in range(n):
        L = landmark_count(i, w, G, B)
        for kk in range(n):
            attended = (i - w < kk <= i) or (kk // B < L)
            if not attended:
                assert np.all(o[i, :, kk] == 0.0)


def test_p4_rows_within_value_hull(oracle_mod):
    rng = np.random.default_rng(11)
    n, G, w, d = 40, 5, 6, 8
    q, k, v = rand_qkv(rng, n, 2, 1, d)
    o, _ = oracle_mod.attn(q, k, v, w, G, 0.5)
    B = n // G
    vlm = v.astype(np.float64).reshape(G, B, 1, d).mean(axis=1)
    for i in range(n):
        rows = [v[j, 0].astype(np.float64) for j in range(max(0, i - w + 1), i + 1)]
        rows += [vlm[l, 0] for l in range(landmark_count(i, w, G, B))]
        rows = np.stack(rows)
        lo, hi = rows.min(axis=0), rows.max(axis=0)
        for h in range(2):
            assert np.all(o[i, h] >= lo - 1e-12) and np.all(o[i, h] <= hi + 1e-12)


# ------------------------------------------------------------------- P5
@pytest.mark.parametrize("n,G,w", [(64, 8, 1), (64, 8, 9), (64, 16, 20), (60, 5, 13)])
def test_p5a_zero_keys_give_uniform_weights(oracle_mod, n, G, w):
    rng = np.random.default_rng(n * w)
    d = 4
    q = rng.standard_normal((n, 2, d)).astype(np.float32)
    k = np.zeros((n, 1, d), dtype=np.float32)
    v = rng.standard_normal((n, 1, d)).astype(np.float32)
    o, l = oracle_mod.attn(q, k, v, w, G, 0.7)
    B = n // G
    vlm = v.astype(np.float64).reshape(G, B, 1, d).mean(axis=1)
    for i in range(n):
        L = landmark_count(i, w, G, B)
        cnt = min(w, i + 1) + L
        assert l[0, i] == pytest.approx(math.log(cnt), abs=1e-13)
        rows = [v[j, 0].astype(np.float64) for j in range(max(0, i - w + 1), i + 1)]
        rows += [vlm[x, 0] for x in range(L)]
        np.testing.assert_allclose(o[i, 0], np.mean(rows, axis=0), rtol=0, atol=1e-12)


def test_p5b_constant_values(oracle_mod):
    rng = np.random.default_rng(2)
    q, k, _ = rand_qkv(rng, 48, 4, 2, 8)
    v = np.full((48, 2, 8), 0.625, dtype=np.float32)
    o, _ = oracle_mod.attn(q, k, v, 7, 6, 0.35)
    np.testing.assert_allclose(o, 0.625, rtol=0, atol=1e-14)


@pytest.mark.parametrize("n,G", [(64, 8), (2048, 16), (96, 96)])
def test_p5c_position_keys_give_block_centres(oracle_mod, n, G):
    k = np.repeat(np.arange(n, dtype=np.float32)[:, None, None], 3, axis=1)
    k = np.repeat(k, 4, axis=2)
    lm = oracle_mod.landmark_pool(k, G)
    B = n // G
    for l in range(G):
        assert np.all(lm[l] == l * B + (B - 1) / 2.0)


def test_p5d_hard_max_limit(oracle_mod):
    """Q[i] = lambda * K[i] with lambda large: row i's output tends to V[i]
    whenever its own key beats every other attended key."""
    rng = np.random.default_rng(4)
    n, G, w, d = 32, 4, 6, 16
    k = rng.standard_normal((n, 1, d)).astype(np.float32)
    v = rng.standard_normal((n, 1, d)).astype(np.float32)
    lam = 200.0
    q = (lam * k).astype(np.float32)
    o, _ = oracle_mod.attn(q, k, v, w, G, 1.0 / math.sqrt(d))
    B = n // G
    klm = k.astype(np.float64).reshape(G, B, 1, d).mean(axis=1)
    checked = 0
    for i in range(n):
        own = float(k[i, 0] @ k[i, 0])
        others = [float(k[i, 0] @ k[j, 0]) for j in range(max(0, i - w + 1), i)]
        others += [float(k[i, 0] @ klm[x, 0]) for x in range(landmark_count(i, w, G, B))]
        if others and own - max(others) < 1.0:
            continue
        np.testing.assert_allclose(o[i, 0], v[i, 0], rtol=0, atol=1e-6)
        checked += 1
    assert checked > n // 2


# ------------------------------------------------------------------- P6
def attended_total_closed_form(n, w, G):
    """sum_i min(w, i+1) + L(i) per head, vectorised closed form."""
    i = np.arange(n, dtype=np.int64)
    win = np.minimum(w, i + 1)
    if G == 0:
        return int(win.sum())
    B = n // G
    lm = np.clip((i - w + 1) // B, 0, G)
    return int(win.sum() + lm.sum())


def test_p6_count_closed_form_matches_set_definition():
    for n, w, G in [(64, 1, 8), (64, 9, 8), (60, 13, 5), (96, 96, 96), (128, 200, 4)]:
        B = n // G
        brute = 0
        for i in range(n):
            brute += sum(1 for j in range(n) if i - w < j <= i)
            brute += sum(1 for l in range(G) if (l + 1) * B <= i - w + 1)
        assert attended_total_closed_form(n, w, G) == brute


def test_p6_oracle_count_via_zero_keys(oracle_mod):
    """With K = 0, exp(lse) is the size of the attended set."""
    n, w, G = 256, 37, 16
    q = np.ones((n, 1, 1), dtype=np.float32)
    k = np.zeros((n, 1, 1), dtype=np.float32)
    _, l = oracle_mod.attn(q, k, k, w, G, 1.0)
    counts = np.rint(np.exp(l[0])).astype(np.int64)
    assert int(counts.sum()) == attended_total_closed_form(n, w, G)


def band_total_closed_form(n, bb, hw):
    i = np.arange(n, dtype=np.int64)
    lo = np.maximum(0, (i // bb - hw) * bb)
    hi = np.minimum(n, (i // bb + hw + 1) * bb)
    return int((hi - lo).sum())


def topk_total_closed_form(n, w, G, top_k, q_block=128):
    """Each row: its window plus min(top_k, candidates of its query block's
    first row) whole blocks."""
    i = np.arange(n, dtype=np.int64)
    B = n // G
    r0 = (i // q_block) * q_block
    cand = np.clip((r0 - w + 1) // B, 0, G)
    return int((np.minimum(w, i + 1) + np.minimum(top_k, cand) * B).sum())


def compressed_total_closed_form(n, w, G, every):
    """Rows c*every - 1 count i + 1 keys, the others min(w, i+1) + L(i)."""
    i = np.arange(n, dtype=np.int64)
    per = np.minimum(w, i + 1) + np.clip((i - w + 1) // (n // G), 0, G)
    glob = np.arange(every - 1, n, every)
    per[glob] = glob + 1
    return int(per.sum())


def test_p6_workload_totals_match_golden():
    with open(os.path.join(GOLDEN, "attended_counts.json")) as f:
        golden = json.load(f)
    for name, wl in WORKLOADS.items():
        if wl.band_block > 0:
            total = band_total_closed_form(wl.n, wl.band_block, wl.band_half)
        elif wl.top_k > 0:
            total = topk_total_closed_form(wl.n, wl.window, wl.G, wl.top_k)
        elif wl.global_every > 0:
            total = compressed_total_closed_form(wl.n, wl.window, wl.G, wl.global_every)
        else:
            total = attended_total_closed_form(wl.n, wl.window, wl.G)
        assert total == golden["per_head"][name], name


def test_p6_page_dot_product_arithmetic():
    """"The Cost of Attention" section counts 64 heads x 1M x 4K = 0.256e12
    window dot products and 64 x 1M x 512 = 0.033e12 landmark ones per layer
    (its 1M = 1e6, 4K = 4e3).  Our exact window count for the million-token
    layer agrees to first order; the landmark count is lower because only
    blocks wholly before the window are visible."""
    wl = WORKLOADS["1m_70b_layer"]
    i = np.arange(wl.n, dtype=np.int64)
    window_total = wl.Hq * int(np.minimum(wl.window, i + 1).sum())
    assert abs(window_total / 0.256e12 - 1.0) < 0.10
    lm_total = wl.Hq * int(np.clip((i - wl.window + 1) // wl.block, 0, wl.G).sum())
    assert 0.3 < lm_total / 0.033e12 < 1.0
    # "Training at 1M+ Token Context", memory paragraph: the KV cache of one
    # layer at 1M tokens, 8 KV heads x 128 x bf16, is about 2 GB per tensor.
    assert abs(wl.n * wl.Hkv * wl.d * 2 / 2**30 - 2.0) < 1e-9


# ------------------------------------------------------------------- band mask
def band_bruteforce(q, k, v, bb, hw, scale):
    """Dense [n, n] band mask built element by element from its definition
    (key block within hw blocks of the row's block), masked softmax."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    n, Hq, d = q.shape
    g = Hq // k.shape[1]
    mask = np.zeros((n, n), dtype=bool)
    for i in range(n):
        for j in range(n):
            mask[i, j] = abs(j // bb - i // bb) <= hw
    out = np.zeros((n, Hq, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        s = np.where(mask, scale * q[:, h] @ k[:, h // g].T, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        e = np.where(mask, np.exp(s - mx), 0.0)
        den = e.sum(axis=1, keepdims=True)
        out[:, h] = (e / den) @ v[:, h // g]
        lse[h] = (mx + np.log(den))[:, 0]
    return out, lse


@pytest.mark.parametrize("n,bb,hw", [(1, 1, 0), (40, 4, 0), (40, 4, 2), (37, 8, 1), (64, 16, 3),
                                     (50, 7, 10)])
def test_band_bruteforce(oracle_mod, n, bb, hw):
    rng = np.random.default_rng(n * bb + hw)
    for (Hq, Hkv), d in itertools.product([(1, 1), (4, 2), (4, 1)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        ro, rl = band_bruteforce(q, k, v, bb, hw, 0.4)
        o, l = oracle_mod.attn_band(q, k, v, bb, hw, 0.4)
        np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


def test_band_wide_enough_is_full_attention(oracle_mod):
    """A half-width covering the sequence is full (non-causal) attention:
    torch SDPA in fp64."""
    rng = np.random.default_rng(9)
    n, Hq, Hkv, d = 96, 4, 2, 16
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    o, _ = oracle_mod.attn_band(q, k, v, 16, 6, 0.25)
    tq = torch.from_numpy(q).double().permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).double().repeat_interleave(2, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).double().repeat_interleave(2, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.25)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_band_count_via_zero_keys(oracle_mod):
    """K = 0: lse = ln of the band's key count; the page's '1/16th' memory
    figure for 16 neighbour blocks out of 256 (a 32K sequence) is the
    first-order ratio (2*8+1)/256."""
    n, bb, hw = 1000, 128, 2
    q = np.ones((n, 1, 1), dtype=np.float32)
    k = np.zeros((n, 1, 1), dtype=np.float32)
    _, l = oracle_mod.attn_band(q, k, k, bb, hw, 1.0)
    i = np.arange(n)
    lo = np.maximum(0, (i // bb - hw) * bb)
    hi = np.minimum(n, (i // bb + hw + 1) * bb)
    np.testing.assert_allclose(np.exp(l[0]), hi - lo, rtol=1e-12)
    assert abs((2 * 8 + 1) / 256 - 1 / 16) < 0.005


# ------------------------------------------------------------------- top-k blocks
def topk_bruteforce(q, k, v, window, G, top_k, scale, qb):
    """numpy: block means, query-block sums, candidate rule, top-k with
    ties to the lower index, dense mask (window or selected block) built
    element by element, masked softmax."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    bs = n // G
    klm = k.reshape(G, bs, Hkv, d).mean(axis=1)
    n_qb = (n + qb - 1) // qb
    chosen = {}
    scores = np.full((n_qb, Hkv, G), -np.inf)
    for t in range(n_qb):
        rows = slice(t * qb, min(n, (t + 1) * qb))
        for c in range(Hkv):
            qs = q[rows, c * g:(c + 1) * g].sum(axis=(0, 1))
            for l in range(G):
                if (l + 1) * bs <= t * qb - window + 1:
                    scores[t, c, l] = qs @ klm[l, c]
            cand = [l for l in range(G) if np.isfinite(scores[t, c, l])]
            order = np.lexsort((np.array(cand), -scores[t, c, cand])) if cand else []
            chosen[(t, c)] = sorted(cand[o] for o in list(order)[:top_k])
    out = np.zeros((n, Hq, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        c = h // g
        mask = np.zeros((n, n), dtype=bool)
        for i in range(n):
            for j in range(n):
                mask[i, j] = (i - window < j <= i) or (j // bs in chosen[(i // qb, c)])
        s = np.where(mask, scale * q[:, h] @ k[:, c].T, -np.inf)
        mx = s.max(axis=1, keepdims=True)
        e = np.where(mask, np.exp(s - mx), 0.0)
        den = e.sum(axis=1, keepdims=True)
        out[:, h] = (e / den) @ v[:, c]
        lse[h] = (mx + np.log(den))[:, 0]
    return scores, chosen, out, lse


@pytest.mark.parametrize("n,G,w,top_k,qb", [(64, 16, 3, 2, 8), (64, 8, 9, 3, 16), (96, 12, 20, 1, 8),
                                            (48, 48, 2, 5, 4), (40, 10, 1, 100, 8)])
def test_topk_bruteforce(oracle_mod, n, G, w, top_k, qb):
    rng = np.random.default_rng(n + G + w + top_k)
    for (Hq, Hkv), d in itertools.product([(2, 1), (4, 2)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        rs, rch, ro, rl = topk_bruteforce(q, k, v, w, G, top_k, 0.4, qb)
        sc = oracle_mod.block_scores(q, k, G, w, q_block=qb)
        np.testing.assert_allclose(sc, rs, rtol=1e-12, atol=1e-12)
        sel, cnt = oracle_mod.select_top_k(sc, top_k)
        for (t, c), blocks in rch.items():
            assert list(sel[t, c, :cnt[t, c]]) == blocks
        o, l = oracle_mod.attn_select(q, k, v, w, G, sel, cnt, 0.4, q_block=qb)
        np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


def test_topk_zero_is_window_attention(oracle_mod):
    rng = np.random.default_rng(21)
    q, k, v = rand_qkv(rng, 64, 4, 2, 8)
    sc = oracle_mod.block_scores(q, k, 8, 5, q_block=16)
    sel, cnt = oracle_mod.select_top_k(sc, 0)
    o, l = oracle_mod.attn_select(q, k, v, 5, 8, sel, cnt, 0.3, q_block=16)
    ro, rl = oracle_mod.attn(q, k, v, 5, 0, 0.3)
    np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


def test_topk_counts_and_ties(oracle_mod):
    """K = 0: every candidate scores 0 (all tied), the lowest indices win,
    and exp(lse) = window size + selected blocks x block size."""
    n, G, w, top_k, qb = 128, 16, 10, 3, 16
    bs = n // G
    q = np.ones((n, 2, 4), dtype=np.float32)
    k = np.zeros((n, 1, 4), dtype=np.float32)
    sc = oracle_mod.block_scores(q, k, G, w, q_block=qb)
    sel, cnt = oracle_mod.select_top_k(sc, top_k)
    for t in range(n // qb):
        n_cand = sum(1 for l in range(G) if (l + 1) * bs <= t * qb - w + 1)
        assert cnt[t, 0] == min(top_k, n_cand)
        assert list(sel[t, 0, :cnt[t, 0]]) == list(range(cnt[t, 0]))
    _, l = oracle_mod.attn_select(q, k, k, w, G, sel, cnt, 1.0, q_block=qb)
    i = np.arange(n)
    expect = np.minimum(w, i + 1) + cnt[i // qb, 0] * bs
    np.testing.assert_allclose(np.exp(l[0]), expect, rtol=1e-12)


def test_topk_planted_block_is_chosen(oracle_mod):
    """Keys of block 2 aligned with every query: block 2 scores highest for
    every query block that may see it."""
    rng = np.random.default_rng(5)
    n, G, w, qb, d = 256, 16, 16, 32, 16
    bs = n // G
    q = (rng.standard_normal((n, 2, d)) * 0.1 + 1.0).astype(np.float32)
    k = (rng.standard_normal((n, 1, d)) * 0.1).astype(np.float32)
    k[2 * bs:3 * bs] += 3.0
    sc = oracle_mod.block_scores(q, k, G, w, q_block=qb)
    sel, cnt = oracle_mod.select_top_k(sc, 1)
    for t in range(n // qb):
        if 3 * bs <= t * qb - w + 1:
            assert cnt[t, 0] == 1 and sel[t, 0, 0] == 2


# ------------------------------------------------------------------- compression tokens + global rows
def compressed_bruteforce(q, k, v, window, block, global_rows, scale):
    """Dense [n, n + n/block] mask built element by element: a global row
    sees every key j <= i; any other row its window and the sub-block means
    whose whole sub-block ends at or before i - w + 1; masked softmax."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    C = n // block
    kc = np.stack([k[c * block:(c + 1) * block].mean(axis=0) for c in range(C)])
    vc = np.stack([v[c * block:(c + 1) * block].mean(axis=0) for c in range(C)])
    gset = set(int(r) for r in global_rows)
    mask = np.zeros((n, n + C), dtype=bool)
    for i in range(n):
        for j in range(n):
            mask[i, j] = j <= i if i in gset else (i - window < j <= i)
        if i not in gset:
            for c in range(C):
                mask[i, n + c] = (c + 1) * block - 1 <= i - window
    out = np.zeros((n, Hq, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        keys = np.concatenate([k[:, h // g], kc[:, h // g]])
        vals = np.concatenate([v[:, h // g], vc[:, h // g]])
        s_ = np.where(mask, scale * q[:, h] @ keys.T, -np.inf)
        mx = s_.max(axis=1, keepdims=True)
        e = np.where(mask, np.exp(s_ - mx), 0.0)
        den = e.sum(axis=1, keepdims=True)
        out[:, h] = (e / den) @ vals
        lse[h] = (mx + np.log(den))[:, 0]
    return out, lse


@pytest.mark.parametrize("n,block,w,glob", [(64, 4, 9, [5, 40, 63]), (64, 8, 1, [0]),
                                            (48, 2, 16, []), (40, 40, 3, [39]),
                                            (96, 4, 20, list(range(0, 96, 7)))])
def test_compressed_bruteforce(oracle_mod, n, block, w, glob):
    rng = np.random.default_rng(n + block + w)
    for (Hq, Hkv), d in itertools.product([(1, 1), (4, 2), (4, 1)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        ro, rl = compressed_bruteforce(q, k, v, w, block, glob, 0.3)
        o, l = oracle_mod.attn_compressed(q, k, v, w, block, glob, 0.3)
        np.testing.assert_allclose(o, ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, rl, rtol=0, atol=1e-12)


def test_compressed_global_rows_are_causal_attention(oracle_mod):
    """Global rows equal torch SDPA with the causal mask (fp64) at those
    rows, whatever the window and compression."""
    rng = np.random.default_rng(21)
    n, Hq, Hkv, d = 128, 4, 2, 16
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    glob = [3, 31, 64, 127]
    o, l = oracle_mod.attn_compressed(q, k, v, 8, 16, glob, 0.25, rows=glob)
    tq = torch.from_numpy(q).double().permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).double().repeat_interleave(2, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).double().repeat_interleave(2, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.25,
                                                           is_causal=True)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy()[glob], rtol=0, atol=1e-12)


def test_compressed_counts_and_page_ratio(oracle_mod):
    """K = 0: exp(lse) counts i + 1 keys on global rows and min(w, i+1) +
    L(i) with 32-token sub-blocks elsewhere; 32-token sub-blocks give the
    page's 256 compression tokens per 8192-token chunk."""
    assert 8192 // 32 == 256
    n, w, block = 1024, 100, 32
    glob = [0, 511, 1023]
    q = np.ones((n, 1, 1), dtype=np.float32)
    k = np.zeros((n, 1, 1), dtype=np.float32)
    _, l = oracle_mod.attn_compressed(q, k, k, w, block, glob, 1.0)
    i = np.arange(n)
    want = np.minimum(w, i + 1) + np.clip((i - w + 1) // block, 0, n // block)
    want[glob] = np.asarray(glob) + 1
    np.testing.assert_allclose(np.exp(l[0]), want, rtol=1e-12)


def test_compressed_gathered_rows_match_indexed_rows(oracle_mod):
    rng = np.random.default_rng(5)
    n = 128
    q, k, v = rand_qkv(rng, n, 4, 2, 8)
    rows = np.array([0, 9, 63, 64, 100, 127])
    glob = [9, 100]
    a = oracle_mod.attn_compressed(q, k, v, 20, 8, glob, 0.3, rows=rows)
    b = oracle_mod.attn_compressed(q[rows], k, v, 20, 8, glob, 0.3, q_positions=rows)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------------------- backward
def dense_torch_grads(q, k, v, dout, window, G, scale):
    """Autograd (fp64) through a dense masked softmax whose mask is built
    element by element from the set definitions and whose landmarks are
    torch block means: an implementation independent of the oracle's
    hand-derived backward."""
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    B = n // G if G else 1
    mask = np.zeros((n, n + G), dtype=bool)
    for i in range(n):
        for j in range(n):
            mask[i, j] = i - window < j <= i
        for l in range(G):
            mask[i, n + l] = (l + 1) * B - 1 <= i - window
    mask_t = torch.from_numpy(mask)
    if G:
        klm = tk.reshape(G, B, Hkv, d).mean(dim=1)
        vlm = tv.reshape(G, B, Hkv, d).mean(dim=1)
        keys, vals = torch.cat([tk, klm]), torch.cat([tv, vlm])
    else:
        keys, vals = tk, tv
    outs = []
    for h in range(Hq):
        s = scale * tq[:, h] @ keys[:, h // g].T
        s = s.masked_fill(~mask_t, float("-inf"))
        outs.append(torch.softmax(s, dim=1) @ vals[:, h // g])
    o = torch.stack(outs, dim=1)
    (o * torch.from_numpy(dout.astype(np.float64))).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("n,G,w", [(16, 4, 3), (16, 0, 5), (24, 6, 1), (32, 8, 9), (12, 12, 2),
                                   (20, 1, 20), (40, 5, 13)])
def test_bwd_matches_dense_autograd(oracle_mod, n, G, w):
    rng = np.random.default_rng(n * 7 + G + w)
    for (Hq, Hkv), d in itertools.product([(1, 1), (4, 2), (4, 1)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        do = rng.standard_normal((n, Hq, d)).astype(np.float32)
        gq, gk, gv = dense_torch_grads(q, k, v, do, w, G, 0.35)
        dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, w, G, 0.35)
        np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-11)
        np.testing.assert_allclose(dk, gk, rtol=0, atol=1e-11)
        np.testing.assert_allclose(dv, gv, rtol=0, atol=1e-11)


def test_bwd_causal_special_case_is_sdpa_backward(oracle_mod):
    """w >= n, G = 0: the gradients of torch SDPA (causal, fp64)."""
    rng = np.random.default_rng(33)
    n, Hq, Hkv, d = 48, 4, 2, 16
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    do = rng.standard_normal((n, Hq, d)).astype(np.float32)
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(2, dim=1).permute(1, 0, 2)[None],
        tv.repeat_interleave(2, dim=1).permute(1, 0, 2)[None], scale=0.25, is_causal=True)
    (o[0].permute(1, 0, 2) * torch.from_numpy(do.astype(np.float64))).sum().backward()
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, n + 3, 0, 0.25)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_central_differences(oracle_mod):
    """A few entries of each gradient against central differences of
    L = sum <dO, O> computed by the forward oracle (fp32 inputs, steps of
    2^-8 that fp32 represents exactly)."""
    rng = np.random.default_rng(4)
    n, Hq, Hkv, d, G, w, sc = 16, 2, 1, 4, 4, 3, 0.5
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    do = rng.standard_normal((n, Hq, d)).astype(np.float32)
    dq, dk, dv = oracle_mod.attn_bwd(q, k, v, do, w, G, sc)

    def loss(q_, k_, v_):
        o, _ = oracle_mod.attn(q_, k_, v_, w, G, sc)
        return float((o * do.astype(np.float64)).sum())

    h = 2.0 ** -8
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for idx in [(0, 0, 0), (5, 0, 2), (15, Hkv - 1, 3), (9, 0, 1)]:
            args = [q.copy(), k.copy(), v.copy()]
            if idx[1] >= args[which].shape[1]:
                continue
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            dn = loss(*args)
            assert abs((up - dn) / (2 * h) - grad[idx]) < 2e-4, (which, idx)


def test_bwd_sum_identities(oracle_mod):
    """Rows of P sum to 1 and rows of dS to 0, so summed over all tokens
    (landmark gradients included) dV of a KV head equals the sum of its
    query heads' dO, and dK sums to zero."""
    rng = np.random.default_rng(8)
    n, Hq, Hkv, d, G, w = 64, 4, 2, 8, 8, 10
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    do = rng.standard_normal((n, Hq, d)).astype(np.float32)
    _, dk, dv = oracle_mod.attn_bwd(q, k, v, do, w, G, 0.3)
    want = do.astype(np.float64).reshape(n, Hkv, Hq // Hkv, d).sum(axis=(0, 2))
    np.testing.assert_allclose(dv.sum(axis=0), want, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, rtol=0, atol=1e-10)


def test_bwd_dq_rows_match_full_backward(oracle_mod):
    rng = np.random.default_rng(12)
    n, Hq, Hkv, d, G, w = 64, 4, 2, 8, 8, 10
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    do = rng.standard_normal((n, Hq, d)).astype(np.float32)
    dq, _, _ = oracle_mod.attn_bwd(q, k, v, do, w, G, 0.3)
    rows = [0, 9, 10, 33, 63]
    np.testing.assert_array_equal(oracle_mod.attn_bwd_dq_rows(q, k, v, do, w, G, 0.3, rows),
                                  dq[rows])


@pytest.mark.parametrize("n,Hq,Hkv,G,w", [(64, 4, 2, 8, 10), (96, 6, 3, 0, 7), (128, 2, 1, 128, 128),
                                           (200, 8, 2, 25, 1), (256, 4, 4, 16, 300)])
def test_bwd_dkdv_keys_match_full_backward(oracle_mod, n, Hq, Hkv, G, w):
    """dK/dV of listed (key, KV head) pairs equal the full backward's rows,
    for every key and head (window keys, landmark blocks seen by many rows,
    by one row, by none; w = 1; w > n; G = 0 and G = n)."""
    rng = np.random.default_rng(n + G + w)
    d = 8
    q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
    do = rng.standard_normal((n, Hq, d)).astype(np.float32)
    _, dk, dv = oracle_mod.attn_bwd(q, k, v, do, w, G, 0.3)
    keys = np.repeat(np.arange(n), Hkv)
    heads = np.tile(np.arange(Hkv), n)
    gk, gv = oracle_mod.attn_bwd_dkdv_keys(q, k, v, do, w, G, 0.3, keys, heads)
    np.testing.assert_allclose(gk, dk.reshape(n * Hkv, d), rtol=0, atol=1e-12)
    np.testing.assert_allclose(gv, dv.reshape(n * Hkv, d), rtol=0, atol=1e-12)
    # an arbitrary subset, in any order, gives the same rows
    pick = rng.permutation(n * Hkv)[: n // 3]
    sk, sv = oracle_mod.attn_bwd_dkdv_keys(q, k, v, do, w, G, 0.3, keys[pick], heads[pick])
    np.testing.assert_array_equal(sk, gk[pick])
    np.testing.assert_array_equal(sv, gv[pick])


def compressed_torch_grads(q, k, v, dout, window, block, global_rows, scale):
    """Autograd (fp64) through the dense mask of the compression-token
    pattern, built element by element as in ``compressed_bruteforce``."""
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    C = n // block
    gset = set(int(r) for r in global_rows)
    mask = np.zeros((n, n + C), dtype=bool)
    for i in range(n):
        for j in range(n):
            mask[i, j] = j <= i if i in gset else (i - window < j <= i)
        if i not in gset:
            for c in range(C):
                mask[i, n + c] = (c + 1) * block - 1 <= i - window
    kc = tk.reshape(C, block, Hkv, d).mean(dim=1)
    vc = tv.reshape(C, block, Hkv, d).mean(dim=1)
    keys, vals = torch.cat([tk, kc]), torch.cat([tv, vc])
    m = torch.from_numpy(mask)
    outs = []
    for h in range(Hq):
        s_ = (scale * tq[:, h] @ keys[:, h // g].T).masked_fill(~m, float("-inf"))
        outs.append(torch.softmax(s_, dim=1) @ vals[:, h // g])
    (torch.stack(outs, dim=1) * torch.from_numpy(dout.astype(np.float64))).sum().backward()
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("n,block,w,glob", [(64, 4, 9, [5, 40, 63]), (48, 8, 1, [0, 47]),
                                            (40, 2, 16, []), (96, 4, 20, list(range(0, 96, 7)))])
def test_compressed_bwd_matches_dense_autograd(oracle_mod, n, block, w, glob):
    rng = np.random.default_rng(n + 3 * block + w)
    for (Hq, Hkv), d in itertools.product([(1, 1), (4, 2)], [4, 8]):
        q, k, v = rand_qkv(rng, n, Hq, Hkv, d)
        do = rng.standard_normal((n, Hq, d)).astype(np.float32)
        ref = compressed_torch_grads(q, k, v, do, w, block, glob, 0.3)
        got = oracle_mod.attn_bwd_compressed(q, k, v, do, w, block, glob, 0.3)
        for g_, r_ in zip(got, ref):
            np.testing.assert_allclose(g_, r_, rtol=0, atol=1e-11)
