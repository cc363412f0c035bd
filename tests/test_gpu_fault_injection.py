"""Failure detection in the tensor-core kernels (forward attention, backward
dK/dV and dQ, global rows), made to happen on purpose without faulting,
trapping or hanging the GPU.

Every mbarrier wait in these kernels is bounded.  The test lowers the bound to
1 ns, which makes every wait that its first, non-blocking probe does not find
complete run out although the copies and MMAs it waits for do complete: the
kernel must then leave its loops, drain what is in flight,
free tensor memory, return, and record MSA_ERR_TIMEOUT in the device status
word -- and the CUDA context must stay usable, which the follow-up launch
with the default bound checks against the oracle.
"""
import numpy as np
import pytest
import torch

from long_context_sparse_landmark_gb300.workloads import Workload, generate
from tests.gpu_helpers import binding, compare, oracle_attention, run_gpu_attention

pytestmark = pytest.mark.gpu


def test_wait_limit_runs_out_and_context_survives():
    B = binding()
    wl = Workload("fault", 8192, 8, 2, 128, 2048, 16, "bf16", seed=21)
    q, k, v = generate(wl, device="cuda")
    assert B.device_status(clear=True) == B.MSA_OK
    try:
        B.set_wait_limit_ns(1)
        run_gpu_attention(q, k, v, wl)
        torch.cuda.synchronize()
        assert B.device_status(clear=True) == B.MSA_ERR_TIMEOUT
    finally:
        B.set_wait_limit_ns(0)
    assert B.device_status(clear=True) == B.MSA_OK
    out, lse = run_gpu_attention(q, k, v, wl)
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == B.MSA_OK
    rows = np.arange(0, wl.n, 97)
    ro, rl = oracle_attention(q, k, v, wl, rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    compare(out.index_select(0, idx).cpu().numpy(), ro, 1e-2, 1e-3, "O after timeout")
    compare(lse.index_select(1, idx).cpu().numpy(), rl, 1e-2, 1e-3, "lse after timeout")


def test_single_cta_kernel_times_out_cleanly():
    """The same for the single-CTA tensor-core kernel, forced where the
    CTA-pair kernel would run."""
    B = binding()
    wl = Workload("fault1", 4096, 8, 2, 128, 1024, 16, "bf16", seed=22)
    q, k, v = generate(wl, device="cuda")
    ref = [t.clone() for t in run_gpu_attention(q, k, v, wl)]
    torch.cuda.synchronize()
    try:
        B.force_single_cta(True)
        got = _timeout_then_clean(B, lambda: run_gpu_attention(q, k, v, wl))
    finally:
        B.force_single_cta(False)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def _timeout_then_clean(B, launch):
    """Run `launch` with every bounded wait cut to 1 ns (expect
    MSA_ERR_TIMEOUT and a clean return), then with the default bound."""
    assert B.device_status(clear=True) == B.MSA_OK
    try:
        B.set_wait_limit_ns(1)
        launch()
        torch.cuda.synchronize()
        assert B.device_status(clear=True) == B.MSA_ERR_TIMEOUT
    finally:
        B.set_wait_limit_ns(0)
    out = launch()
    torch.cuda.synchronize()
    assert B.device_status(clear=True) == B.MSA_OK
    return out


def test_fused_ring_rounds_time_out_cleanly():
    """Fused ring rounds (a partial round, then running merges whose epilogue
    loads, combines and stores O through shared memory) leave cleanly when
    their waits run out; rounds run afresh afterwards give the same bits."""
    import long_context_sparse_landmark_gb300.api as api
    B = binding()
    wl = Workload("fault_ring", 4096, 8, 2, 128, 4096, 0, "bf16", seed=26)
    q, k, v = generate(wl, device="cuda")
    ref = [t.clone() for t in api.ring_attention(q, k, v, 4, fused=True)]
    torch.cuda.synchronize()
    got = _timeout_then_clean(B, lambda: api.ring_attention(q, k, v, 4, fused=True))
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_backward_kernels_time_out_cleanly():
    """The dK/dV (both modes) and dQ kernels leave their pipelines, drain and
    free TMEM when their waits run out; the next call is exact again."""
    import long_context_sparse_landmark_gb300.api as api
    B = binding()
    wl = Workload("fault_bwd", 4096, 8, 2, 128, 512, 16, "bf16", seed=23)
    q, k, v = generate(wl, device="cuda")
    out, lse = api.msa_attention(q, k, v, wl.window, wl.G, wl.scale, out_dtype=torch.float32)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(24)
    do = torch.randn(q.shape, generator=gen, device="cuda").to(torch.bfloat16)
    torch.cuda.synchronize()
    ref = [t.clone() for t in api.msa_attention_backward(q, k, v, out, lse, do, wl.window,
                                                         wl.G, wl.scale,
                                                         grad_dtype=torch.float32)]
    torch.cuda.synchronize()
    got = _timeout_then_clean(B, lambda: api.msa_attention_backward(
        q, k, v, out, lse, do, wl.window, wl.G, wl.scale, grad_dtype=torch.float32))
    for g, r in zip(got, ref):
        assert torch.equal(g, r)


def test_global_rows_kernel_times_out_cleanly():
    B = binding()
    wl = Workload("fault_gr", 8192, 16, 2, 128, 1, 0, "bf16", seed=25)
    q, k, v = generate(wl, device="cuda")
    rows = torch.tensor([8191, 4000, 77, 5000], dtype=torch.int64, device="cuda")
    ws = torch.empty((B.global_rows_workspace_size(wl.n, 4, wl.Hq, wl.Hkv, wl.d),),
                     dtype=torch.uint8, device="cuda")

    def launch():
        out = torch.zeros((wl.n, wl.Hq, wl.d), dtype=torch.float32, device="cuda")
        lse = torch.zeros((wl.Hq, wl.n), dtype=torch.float32, device="cuda")
        B.attn_fwd_global_rows(q, k, v, rows, out, lse, wl.scale, ws)
        return out, lse

    ref = launch()
    torch.cuda.synchronize()
    got = _timeout_then_clean(B, launch)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
