"""User-facing calls: allocate outputs with torch, run libmsa's kernels.

``msa_attention`` is the whole window + landmark forward (pool, then fused
attention); ``ring_attention`` is the one-GPU emulation of a Ring Attention
layer (per-chunk partials, then the LSE merge).  Both only marshal
arguments: every arithmetic step runs in libmsa's CUDA kernels.
"""
from __future__ import annotations

import math
import warnings

import torch

from . import _binding as B


class CudaCorePathWarning(RuntimeWarning):
    """A bf16 attention runs on the CUDA-core (fp32 FFMA) kernel, many times
    slower than the tensor-core kernels, because of its shape."""


_warned = set()


def _check_tensor_cores(q: torch.Tensor, Hkv: int, topk_landmarks: int | None = None):
    """Warn (once per shape) when bf16 input is routed to the CUDA-core
    kernel: d other than 128, or (top-k) a key block that is not a whole
    number of 128-key tiles.  fp32 input always runs there, by design."""
    if q.dtype != torch.bfloat16:
        return
    n, Hq, d = q.shape
    if topk_landmarks is None:
        tc = B.uses_tensor_cores(Hq, Hkv, d, q.dtype)
    else:
        tc = B.topk_uses_tensor_cores(n, Hq, Hkv, d, topk_landmarks, q.dtype)
    key = (n if topk_landmarks is not None else 0, Hq, Hkv, d, topk_landmarks)
    if not tc and key not in _warned:
        _warned.add(key)
        why = (f"d={d} (the tensor-core kernels take d=128)" if d != 128 else
               f"key blocks of {n // max(topk_landmarks, 1)} tokens are not a multiple of 128")
        warnings.warn(f"bf16 attention on the CUDA-core kernel: {why}", CudaCorePathWarning,
                      stacklevel=3)


def landmarks(k: torch.Tensor, v: torch.Tensor, n_landmarks: int, stream=None):
    """Block-mean landmarks K_lm, V_lm [G, Hkv, d] of k, v [n, Hkv, d]."""
    n, Hkv, d = k.shape
    k_lm = torch.empty((n_landmarks, Hkv, d), dtype=k.dtype, device=k.device)
    v_lm = torch.empty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm, stream=stream)
    return k_lm, v_lm


def msa_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int,
                  n_landmarks: int, scale: float | None = None,
                  out_dtype: torch.dtype | None = None, stream=None):
    """Window + landmark attention forward.

    q [n, Hq, d], k/v [n, Hkv, d] (bf16 or fp32, same dtype, on one GPU).
    Returns (out [n, Hq, d] in ``out_dtype`` (default: q's dtype),
    lse [Hq, n] fp32).
    """
    n, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty((n, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
    if n_landmarks > 0:
        k_lm, v_lm = landmarks(k, v, n_landmarks, stream=stream)
    else:
        k_lm = v_lm = None
    _check_tensor_cores(q, k.shape[1])
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, window, n_landmarks, scale, stream=stream)
    return out, lse


def band_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, band_block: int = 128,
                   band_half: int = 8, scale: float | None = None,
                   out_dtype: torch.dtype | None = None, stream=None):
    """Block-band attention (each band_block-token block attends the blocks
    within band_half of it, both sides).  Returns (out, lse)."""
    n, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty((n, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
    _check_tensor_cores(q, k.shape[1])
    B.attn_fwd_band(q, k, v, out, lse, band_block, band_half, scale, stream=stream)
    return out, lse


def topk_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int,
                   n_landmarks: int, top_k: int, scale: float | None = None,
                   out_dtype: torch.dtype | None = None, stream=None):
    """Window + top-k selected key blocks (msa_attn_fwd_topk; the workspace
    is a torch allocation).  Returns (out, lse)."""
    n, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty((n, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
    nbytes = B.topk_workspace_size(n, k.shape[1], d, n_landmarks, top_k, q.dtype)
    ws = torch.empty((nbytes,), dtype=torch.uint8, device=q.device)
    _check_tensor_cores(q, k.shape[1], n_landmarks)
    B.attn_fwd_topk(q, k, v, out, lse, window, n_landmarks, top_k, scale, ws, stream=stream)
    return out, lse


def compressed_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int,
                         block: int, global_rows: torch.Tensor, scale: float | None = None,
                         out_dtype: torch.dtype | None = None, stream=None):
    """Compression tokens + global query rows: every row attends its window
    and the means of the `block`-token sub-blocks wholly before it
    (msa_landmark_pool + msa_attn_fwd with n / block landmarks); the rows in
    `global_rows` (int64 positions on the device) then attend every key
    j <= their position (msa_attn_fwd_global_rows).  Returns (out, lse)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    G = n // block
    k_lm = torch.empty((G, Hkv, d), dtype=k.dtype, device=k.device)
    v_lm = torch.empty_like(k_lm)
    B.landmark_pool(k, v, k_lm, v_lm, stream=stream)
    out = torch.empty((n, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
    _check_tensor_cores(q, Hkv)
    B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, window, G, scale, stream=stream)
    if global_rows.numel() > 0:
        ws = torch.empty((B.global_rows_workspace_size(n, global_rows.numel(), Hq, Hkv, d),),
                         dtype=torch.uint8, device=q.device)
        B.attn_fwd_global_rows(q, k, v, global_rows, out, lse, scale, ws, stream=stream)
    return out, lse


def ring_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, n_chunks: int,
                   window: int | None = None, scale: float | None = None,
                   out_dtype: torch.dtype | None = None, fused: bool = True, stream=None):
    """Causal (windowed) attention computed as a Ring Attention layer would:
    the KV sequence is cut into ``n_chunks`` contiguous chunks and each
    chunk's partial is aggregated by log-sum-exp.  ``fused`` merges every
    chunk into a running fp32 result inside the attention kernel (the
    partials never reach HBM); otherwise all partials are written and merged
    by ``msa_lse_merge`` at the end.  Returns (out, lse); with ``fused`` the
    output is fp32 (the running accumulator)."""
    n, Hq, d = q.shape
    if n % n_chunks != 0:
        raise ValueError("n must be a multiple of n_chunks")
    window = n if window is None else window
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    c = n // n_chunks
    _check_tensor_cores(q, k.shape[1])
    if fused:
        # The first round writes the running result (rows with no key get
        # lse = -inf, which later rounds treat as empty); the others merge.
        out = torch.empty((n, Hq, d), dtype=torch.float32, device=q.device)
        lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
        B.attn_fwd_partial(q, k[:c], v[:c], out, lse, 0, 0, window, scale, stream=stream)
        for p in range(1, n_chunks):
            B.attn_fwd_partial_merge(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], out, lse, 0,
                                     p * c, window, scale, stream=stream)
        return out, lse
    o_parts = [torch.empty((n, Hq, d), dtype=torch.float32, device=q.device)
               for _ in range(n_chunks)]
    lse_parts = [torch.empty((Hq, n), dtype=torch.float32, device=q.device)
                 for _ in range(n_chunks)]
    for p in range(n_chunks):
        B.attn_fwd_partial(q, k[p * c:(p + 1) * c], v[p * c:(p + 1) * c], o_parts[p],
                           lse_parts[p], 0, p * c, window, scale, stream=stream)
    out = torch.empty((n, Hq, d), dtype=out_dtype or q.dtype, device=q.device)
    lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
    B.lse_merge(o_parts, lse_parts, out, lse, stream=stream)
    return out, lse


def msa_attention_backward(q, k, v, out, lse, dout, window: int, n_landmarks: int,
                           scale: float | None = None, grad_dtype: torch.dtype | None = None,
                           landmarks_kv=None, stream=None):
    """Gradients (dq, dk, dv) of sum <dout, out> for the window + landmark
    forward whose (out, lse) are given; bf16 inputs, d = 128.  The landmark
    keys/values are pooled again unless ``landmarks_kv`` passes the
    forward's."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if n_landmarks > 0:
        k_lm, v_lm = landmarks_kv if landmarks_kv is not None else landmarks(
            k, v, n_landmarks, stream=stream)
    else:
        k_lm = v_lm = None
    gdt = grad_dtype or q.dtype
    dq = torch.empty((n, Hq, d), dtype=gdt, device=q.device)
    dk = torch.empty((n, Hkv, d), dtype=gdt, device=q.device)
    dv = torch.empty_like(dk)
    ws = torch.empty((B.attn_bwd_workspace_size(n, Hq, Hkv, d, n_landmarks),), dtype=torch.uint8,
                     device=q.device)
    B.attn_bwd(q, k, v, k_lm, v_lm, out, lse, dout.contiguous(), dq, dk, dv, window,
               n_landmarks, scale, ws, stream=stream)
    return dq, dk, dv


def compressed_attention_backward(q, k, v, out, lse, dout, window: int, block: int,
                                  global_rows: torch.Tensor, scale: float | None = None,
                                  grad_dtype: torch.dtype | None = None, stream=None):
    """Gradients (dq, dk, dv) of sum <dout, out> for ``compressed_attention``
    (whose out, lse are given): bf16 inputs, d = 128."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    G = n // block
    k_lm, v_lm = landmarks(k, v, G, stream=stream)
    gdt = grad_dtype or q.dtype
    dq = torch.empty((n, Hq, d), dtype=gdt, device=q.device)
    dk = torch.empty((n, Hkv, d), dtype=gdt, device=q.device)
    dv = torch.empty_like(dk)
    ws = torch.empty((B.attn_bwd_global_rows_workspace_size(n, global_rows.numel(), Hq, Hkv, d,
                                                           G),),
                     dtype=torch.uint8, device=q.device)
    B.attn_bwd_global_rows(q, k, v, k_lm, v_lm, out, lse, dout.contiguous(), global_rows, dq,
                           dk, dv, window, G, scale, ws, stream=stream)
    return dq, dk, dv


class _MSAAttention(torch.autograd.Function):
    """Window + landmark attention as a differentiable op (libmsa forward
    and backward kernels)."""

    @staticmethod
    def forward(ctx, q, k, v, window, n_landmarks, scale):
        n, Hq, d = q.shape
        out = torch.empty_like(q)
        lse = torch.empty((Hq, n), dtype=torch.float32, device=q.device)
        if n_landmarks > 0:
            k_lm, v_lm = landmarks(k, v, n_landmarks)
        else:
            k_lm = v_lm = None
        B.attn_fwd(q, k, v, k_lm, v_lm, out, lse, window, n_landmarks, scale)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.lm = (k_lm, v_lm)
        ctx.cfg = (window, n_landmarks, scale)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        window, n_landmarks, scale = ctx.cfg
        dq, dk, dv = msa_attention_backward(
            q, k, v, out, lse, dout.to(q.dtype), window, n_landmarks, scale,
            landmarks_kv=ctx.lm if n_landmarks > 0 else None)
        return dq, dk, dv, None, None, None


def msa_attention_trainable(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, window: int,
                            n_landmarks: int, scale: float | None = None) -> torch.Tensor:
    """Differentiable window + landmark attention (bf16, d = 128): returns
    out [n, Hq, d]; ``out.backward(g)`` runs msa_attn_bwd."""
    scale = 1.0 / math.sqrt(q.shape[2]) if scale is None else scale
    return _MSAAttention.apply(q, k, v, window, n_landmarks, scale)


_copy_streams = {}


def _streams_for(dev: torch.device):
    """Two copy streams per device, made once and reused by every call."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _copy_streams:
        _copy_streams[key] = (torch.cuda.Stream(key), torch.cuda.Stream(key))
    return _copy_streams[key]


def msa_attention_host(hq: torch.Tensor, hk: torch.Tensor, hv: torch.Tensor, window: int,
                       n_landmarks: int, scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, chunk_rows: int | None = None,
                       device=None):
    """Window + landmark attention on host (pinned) tensors: msa_attn_fwd_host.

    The library streams K, V and Q through the device in row chunks (default
    about n/32 rows, at least 4096), pools each chunk's landmarks, attends
    its rows and copies O back, the copies overlapping the kernels; this
    function allocates the device workspace and the pinned outputs and
    passes the current stream and two reused copy streams.  Returns host
    (out [n, Hq, d] in q's dtype, lse [Hq, n] fp32), complete when the call
    returns.
    """
    dev = torch.device(device) if device is not None else torch.device("cuda")
    n, Hq, d = hq.shape
    Hkv = hk.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty((n, Hq, d), dtype=hq.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty((Hq, n), dtype=torch.float32, pin_memory=True)
    rows = 0 if chunk_rows is None else int(chunk_rows)
    _check_tensor_cores(hq, Hkv)
    with torch.cuda.device(dev):
        ws = torch.empty((B.host_workspace_size(n, Hq, Hkv, d, int(n_landmarks), rows, hq.dtype,
                                                out.dtype),), dtype=torch.uint8, device=dev)
        s_in, s_out = _streams_for(dev)
        B.attn_fwd_host(hq, hk, hv, out, lse, window, int(n_landmarks), scale, rows, ws,
                        stream=torch.cuda.current_stream(dev), copy_in=s_in, copy_out=s_out)
    return out, lse


class SparseLandmarkAttention(torch.nn.Module):
    """Window + landmark attention as a module, configured like the pages'
    Flash-MSA layer ("Scaling GPU Cluster for Million Token Context": a
    local window and a number of global landmark tokens, set by the
    SPARSE_WINDOW and SPARSE_GLOBAL_TOKENS environment variables in its
    launch script).  ``window`` and ``num_global`` default to those
    variables, else 4096 and 512.  Unlike the pages' sketch, which returns
    the local and global contributions separately, the result is one
    attention over both sets (one softmax, one lse).

    forward(q, k, v): q [n, Hq, d] or [batch, n, Hq, d], k and v with Hkv
    heads; num_global must divide n.  Differentiable (msa_attn_bwd) for bf16
    inputs with d = 128 when gradients are required.
    """

    def __init__(self, window: int | None = None, num_global: int | None = None,
                 scale: float | None = None):
        super().__init__()
        import os
        self.window = int(os.environ.get("SPARSE_WINDOW", "4096")) if window is None else int(window)
        self.num_global = (int(os.environ.get("SPARSE_GLOBAL_TOKENS", "512"))
                           if num_global is None else int(num_global))
        self.scale = scale
        if self.window < 1 or self.num_global < 0:
            raise ValueError("window must be >= 1 and num_global >= 0")

    def _one(self, q, k, v):
        n = q.shape[0]
        if self.num_global and n % self.num_global != 0:
            raise ValueError(f"num_global={self.num_global} must divide the sequence length {n}")
        scale = 1.0 / math.sqrt(q.shape[2]) if self.scale is None else self.scale
        if torch.is_grad_enabled() and (q.requires_grad or k.requires_grad or v.requires_grad):
            return msa_attention_trainable(q, k, v, self.window, self.num_global, scale)
        return msa_attention(q, k, v, self.window, self.num_global, scale)[0]

    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
        if q.dim() == 3:
            return self._one(q, k, v)
        return torch.stack([self._one(q[b], k[b], v[b]) for b in range(q.shape[0])])
