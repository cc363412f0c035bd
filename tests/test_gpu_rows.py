"""Query-row ranges (msa_attn_fwd_rows) and the host streaming entry point
(msa_attn_fwd_host, and msa_attention_host above it): row chunks reproduce the whole-sequence call bit for
bit when they start on 128-row tiles (the same tiles run the same
arithmetic), ragged chunks match the oracle at their global positions, and
the host API returns exactly the device API's results (K/V and landmarks
streamed per chunk when chunks are whole landmark blocks, copied whole
first otherwise; ragged last chunks; no landmarks)."""
import numpy as np
import pytest
import torch

import oracle
from long_context_sparse_landmark_gb300.workloads import (WORKLOADS, Workload, generate,
                                                          to_numpy_bits)
from tests.gpu_helpers import (binding, compare, gempty, gempty_like, gfull, gfull_like,
                               run_gpu_attention, tol)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_row_chunks_equal_whole_call(dt, d):
    B = binding()
    wl = Workload("rows", 4096, 8, 2, d, 700, 16, dt, seed=41)
    q, k, v = generate(wl, device=DEV)
    ref_o, ref_l = run_gpu_attention(q, k, v, wl)
    k_lm = gempty((wl.G, wl.Hkv, d), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)
    out = gfull_like(ref_o, float("nan"))
    lse = gfull_like(ref_l, float("nan"))
    for r0 in range(0, wl.n, 1024):
        B.attn_fwd_rows(q[r0:r0 + 1024], k, v, k_lm, v_lm, out[r0:r0 + 1024], lse, r0,
                        wl.window, wl.G, wl.scale)
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)


@pytest.mark.parametrize("dt,d", [("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("q_start,n_q", [(1000, 777), (0, 1), (4095, 1), (3, 300)])
def test_ragged_row_range_matches_oracle(dt, d, q_start, n_q):
    B = binding()
    wl = Workload("rr", 4096, 4, 1, d, 300, 32, dt, seed=q_start + n_q)
    q, k, v = generate(wl, device=DEV)
    k_lm = gempty((wl.G, wl.Hkv, d), dtype=k.dtype, device=DEV)
    v_lm = gempty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm)
    qr = q[q_start:q_start + n_q].contiguous()
    out = gempty((n_q, wl.Hq, d), dtype=torch.float32, device=DEV)
    lse = gfull((wl.Hq, wl.n), float("nan"), dtype=torch.float32, device=DEV)
    B.attn_fwd_rows(qr, k, v, k_lm, v_lm, out, lse, q_start, wl.window, wl.G, wl.scale)
    torch.cuda.synchronize()
    rows = np.arange(q_start, q_start + n_q)
    ro, rl = oracle.attn(to_numpy_bits(qr), to_numpy_bits(k), to_numpy_bits(v), wl.window,
                         wl.G, wl.scale, q_positions=rows)
    mx, mean = tol(dt)
    compare(out.cpu().numpy(), ro, mx, mean, "row range O")
    got_l = lse.cpu().numpy()
    compare(got_l[:, q_start:q_start + n_q], rl, mx, mean, "row range lse")
    others = np.ones(wl.n, dtype=bool)
    others[q_start:q_start + n_q] = False
    assert np.isnan(got_l[:, others]).all(), "lse columns outside the range were written"


_L = pytest.mark.large


@pytest.mark.parametrize("name,chunk", [("32k_outliers", 4096),
                                        pytest.param("128k_70b_layer", 16384, marks=_L),
                                        ("pr1_2k", 300), ("32k_outliers", 4160),
                                        pytest.param("ring_128k", 20000, marks=_L),
                                        pytest.param("128k_70b_layer", None, marks=_L),
                                        pytest.param("128k_70b_layer", 4224, marks=_L)])
def test_host_api_equals_device_api(name, chunk):
    """msa_attn_fwd_host through the Python API (copy streams, pinned
    buffers): whole landmark blocks per chunk (K/V streamed), chunks that
    are not (K/V copied and pooled whole first: 4224 rows at B = 256),
    ragged last chunks, no landmarks, the fp32 CUDA-core path."""
    import long_context_sparse_landmark_gb300.api as api
    wl = WORKLOADS[name]
    q, k, v = generate(wl, device=DEV)
    ref_o, ref_l = api.msa_attention(q, k, v, wl.window, wl.G, wl.scale)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho, hl = api.msa_attention_host(hq, hk, hv, wl.window, wl.G, wl.scale, chunk_rows=chunk)
    assert torch.equal(ho, ref_o.cpu()) and torch.equal(hl, ref_l.cpu())


@pytest.mark.parametrize("dt,d,n,G,w,chunk", [("bf16", 128, 3000, 12, 700, 640),
                                              ("f32", 64, 2048, 16, 256, 128),
                                              ("bf16", 128, 1000, 0, 1000, 0)])
def test_host_entry_point_one_stream(dt, d, n, G, w, chunk):
    """The C entry point called directly with no copy streams (everything on
    one stream) and pageable host memory: same bits as msa_attn_fwd."""
    B = binding()
    wl = Workload("host1", n, 8, 2, d, w, G, dt, seed=n + G)
    q, k, v = generate(wl, device=DEV)
    ref_o, ref_l = run_gpu_attention(q, k, v, wl)
    hq, hk, hv = (t.cpu() for t in (q, k, v))
    ho = torch.full((n, 8, d), float("nan"))
    hl = torch.full((8, n), float("nan"))
    ws = gempty((B.host_workspace_size(n, 8, 2, d, G, chunk, q.dtype, torch.float32),),
                dtype=torch.uint8, device=DEV)
    B.attn_fwd_host(hq, hk, hv, ho, hl, w, G, wl.scale, chunk, ws)
    assert B.device_status() == 0
    assert torch.equal(ho, ref_o.cpu()) and torch.equal(hl, ref_l.cpu())


def test_module_batches_and_gradients():
    """SparseLandmarkAttention over a batch of 2 equals per-sequence calls;
    with gradients it runs the backward kernels."""
    import long_context_sparse_landmark_gb300.api as api
    from long_context_sparse_landmark_gb300 import SparseLandmarkAttention
    wl = Workload("mod", 2048, 8, 2, 128, 300, 16, "bf16", seed=91)
    qs, ks, vs = zip(*(generate(wl, device=DEV, seed=s) for s in (91, 92)))
    q, k, v = (torch.stack(t) for t in (qs, ks, vs))
    m = SparseLandmarkAttention(window=wl.window, num_global=wl.G)
    with torch.no_grad():
        out = m(q, k, v)
    for b in range(2):
        ref, _ = api.msa_attention(q[b], k[b], v[b], wl.window, wl.G)
        assert torch.equal(out[b], ref)
    qa = q.clone().requires_grad_(True)
    out = m(qa, k, v)
    out.float().sum().backward()
    torch.cuda.synchronize()
    assert qa.grad is not None and torch.isfinite(qa.grad.float()).all()
    assert binding().device_status() == 0
