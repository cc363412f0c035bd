"""msa_attn_fwd_topk_noalloc: the one-call top-k path on the library's fixed
per-device scratch gives the results of msa_attn_fwd_topk with a caller
workspace, call after call, and refuses sizes its scratch cannot hold.

The test first runs a larger shape, which writes more of the scratch than
any later case, so every later call starts on bytes left by another call;
it does not depend on what ran before it in the process."""
import ctypes

import numpy as np
import pytest
import torch

from long_context_sparse_landmark_gb300.workloads import Workload, generate
from tests.gpu_helpers import binding, compare, gempty, gfull, tol

DEV = "cuda"
SCRATCH_BYTES = 16 << 20

# Written first: 32K tokens, 128 blocks, top-48 over 4 KV heads fills more of
# the scratch (block-mean keys, selection, counts) than any case below.
LARGER = ("bf16", 128, 32768, 128, 1024, 48, 16, 4)

CASES = [
    # dt, d, n, G, w, top_k, Hq, Hkv   (tensor-core path, then CUDA-core paths)
    ("bf16", 128, 8192, 32, 1024, 6, 16, 2),
    ("f32", 64, 1000, 8, 100, 2, 4, 1),
    ("bf16", 64, 2048, 16, 128, 16, 6, 6),
]


def _with_workspace(q, k, v, wl, out_dtype):
    B = binding()
    out = gempty((wl.n, wl.Hq, wl.d), dtype=out_dtype, device=DEV)
    lse = gempty((wl.Hq, wl.n), dtype=torch.float32, device=DEV)
    ws = gempty((B.topk_workspace_size(wl.n, wl.Hkv, wl.d, wl.G, wl.top_k, q.dtype),),
                dtype=torch.uint8, device=DEV)
    B.attn_fwd_topk(q, k, v, out, lse, wl.window, wl.G, wl.top_k, wl.scale, ws)
    return out, lse


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    B = binding()
    big = B.topk_workspace_size(LARGER[2], LARGER[7], LARGER[1], LARGER[3], LARGER[5],
                                torch.bfloat16)
    for dt, d, n, G, w, top_k, Hq, Hkv in CASES:
        dtype = torch.bfloat16 if dt == "bf16" else torch.float32
        assert B.topk_workspace_size(n, Hkv, d, G, top_k, dtype) < big
    for dt, d, n, G, w, top_k, Hq, Hkv in [LARGER] + CASES:
        wl = Workload("noalloc", n, Hq, Hkv, d, w, G, dt, seed=n + G, top_k=top_k)
        q, k, v = generate(wl, device=DEV)
        ref_o, ref_l = _with_workspace(q, k, v, wl, torch.float32)
        torch.cuda.synchronize()
        mx, mean = tol(dt)
        for call in range(2):
            out = gfull((n, Hq, d), float("nan"), dtype=torch.float32, device=DEV)
            lse = gfull((Hq, n), float("nan"), dtype=torch.float32, device=DEV)
            B.attn_fwd_topk_noalloc(q, k, v, out, lse, w, G, top_k, wl.scale)
            torch.cuda.synchronize()
            assert B.device_status() == 0
            compare(out.cpu().numpy(), ref_o.cpu().numpy(), mx, mean, f"noalloc O call {call}")
            compare(lse.cpu().numpy(), ref_l.cpu().numpy(), mx, mean, f"noalloc lse call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Sizes whose workspace exceeds the fixed scratch are refused with
    MSA_ERR_UNSUPPORTED before anything runs (host-side, no GPU needed)."""
    from long_context_sparse_landmark_gb300 import build, _binding
    lib = _binding.load_library(build.build())
    size = lib.msa_attn_fwd_topk_workspace_size
    good = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    f = lib.msa_attn_fwd_topk_noalloc
    # 2^21 tokens, 8 KV heads, 1024 blocks, top-64: 64 MiB of selection alone
    n, Hkv, d, G, top_k = 1 << 21, 8, 128, 1024, 64
    assert size(n, Hkv, d, G, top_k, 1) > SCRATCH_BYTES
    rc = f(good, good, good, good, good, n, 64, Hkv, d, 1024, G, top_k, ctypes.c_float(0.1),
           1, 0, None)
    assert rc == 2  # MSA_ERR_UNSUPPORTED
    assert b"scratch" in lib.msa_last_error_string()
    # The 1M-token layer with 512 blocks and top-50 fits.
    assert size(1 << 20, 8, 128, 512, 50, 1) <= SCRATCH_BYTES
