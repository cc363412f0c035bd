"""Failure detection in the tensor-core kernel, made to happen on purpose
without faulting, trapping or hanging the GPU.

Every mbarrier wait in the kernel is bounded.  The test lowers the bound to
1 ns so that waits run out although the copies and MMAs they wait for do
complete: the kernel must then leave its loops, drain what is in flight,
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
