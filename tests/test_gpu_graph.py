"""CUDA graphs: the entry points enqueue work on the caller's stream and
neither allocate nor synchronise, so a step made of them can be captured
once and replayed.  A captured pool + forward step and a captured ring layer
(eight rounds merged in the epilogue) replay to the bits of the same calls
made eagerly, with new inputs copied into the captured buffers between
replays."""
import pytest
import torch

from long_context_sparse_landmark_gb300.workloads import Workload, generate
from tests.gpu_helpers import binding

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _same(a, b):
    return all(torch.equal(_bits(x), _bits(y)) for x, y in zip(a, b))


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (4, 4)])
def test_forward_step_replays_from_a_graph(Hq, Hkv):
    """Pool + attention captured on a side stream (the pair kernel for a
    group of eight, the single-CTA kernel for one head per KV head)."""
    B = binding()
    wl = Workload("graph", 8192, Hq, Hkv, 128, 1024, 32, "bf16", seed=31)
    q, k, v = generate(wl, device=DEV)
    k_lm = torch.empty((wl.G, Hkv, 128), dtype=k.dtype, device=DEV)
    v_lm = torch.empty_like(k_lm)
    out = torch.empty((wl.n, Hq, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((Hq, wl.n), device=DEV)

    def step(stream):
        B.landmark_pool(k, v, k_lm, v_lm, stream=stream)
        B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, wl.window, wl.G, wl.scale, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(side)  # loads the device code and sets function attributes before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = (out.clone(), lse.clone())

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(torch.cuda.current_stream())
    out.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert _same((out, lse), eager), "graph replay differs from the eager step"

    # new inputs in the captured buffers: the replay follows them
    q2, k2, v2 = generate(Workload("graph2", 8192, Hq, Hkv, 128, 1024, 32, "bf16", seed=32),
                          device=DEV)
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager2 = (out.clone(), lse.clone())
    assert not _same(eager2, eager)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert B.device_status() == 0
    assert _same((out, lse), eager2), "replay on new inputs differs from the eager step"


def test_ring_layer_replays_from_a_graph():
    """One partial and seven rounds merged into the running result, captured
    as one graph (16 launches' worth of host work replaced by one replay)."""
    B = binding()
    wl = Workload("graph_ring", 8192, 8, 2, 128, 8192, 0, "bf16", seed=33)
    q, k, v = generate(wl, device=DEV)
    c = wl.n // 8
    o = torch.empty((wl.n, wl.Hq, 128), device=DEV)
    l_ = torch.empty((wl.Hq, wl.n), device=DEV)

    def layer(stream):
        B.attn_fwd_partial(q, k[:c], v[:c], o, l_, 0, 0, wl.window, wl.scale, stream=stream)
        for p in range(1, 8):
            B.attn_fwd_partial_merge(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], o, l_, 0,
                                     p * c, wl.window, wl.scale, stream=stream)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = (o.clone(), l_.clone())

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(torch.cuda.current_stream())
    for _ in range(2):
        o.fill_(float("nan"))
        l_.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert B.device_status() == 0
        assert _same((o, l_), eager), "ring layer replay differs from the eager layer"
