"""ctypes binding of libmsa's C ABI (include/msa.h), argument marshalling only.

Each function here takes torch tensors, checks device/dtype/contiguity,
and passes raw device pointers plus the current CUDA stream to the C entry
point of the same name.  All arithmetic runs in libmsa's CUDA kernels; if
the library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MSA_DEBUG_BOUNDS=1 loads the bounds-checked build (libmsa_debug.so, from
# build.build(debug_bounds=True)) instead of the normal library.
DEBUG_BOUNDS = os.environ.get("MSA_DEBUG_BOUNDS") == "1"
LIB_PATH = os.path.join(_PKG, "libmsa_debug.so" if DEBUG_BOUNDS else "libmsa.so")

MSA_OK, MSA_ERR_INVALID_ARG, MSA_ERR_UNSUPPORTED, MSA_ERR_CUDA, MSA_ERR_TIMEOUT = range(5)
MSA_F32, MSA_BF16 = 0, 1
MAX_MERGE_PARTS = 64

# Every symbol include/msa.h declares.
EXPORTS = ("msa_version", "msa_last_error_string", "msa_landmark_pool", "msa_attn_fwd",
           "msa_attn_fwd_rows", "msa_attn_fwd_host", "msa_attn_fwd_host_workspace_size",
           "msa_attn_fwd_band", "msa_block_select", "msa_attn_fwd_select",
           "msa_attn_fwd_topk_workspace_size", "msa_attn_fwd_topk", "msa_attn_fwd_topk_noalloc",
           "msa_attn_fwd_global_rows", "msa_attn_fwd_global_rows_workspace_size",
           "msa_attn_bwd", "msa_attn_bwd_workspace_size", "msa_attn_bwd_global_rows",
           "msa_attn_bwd_global_rows_workspace_size", "msa_attn_fwd_partial",
           "msa_attn_fwd_partial_merge", "msa_lse_merge",
           "msa_attn_uses_tensor_cores", "msa_attn_fwd_topk_uses_tensor_cores",
           "msa_debug_bounds_build", "msa_device_status", "msa_debug_set_wait_limit_ns",
           "msa_debug_force_single_cta", "msa_debug_set_max_clusters")


class MsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"msa status {status}: {msg}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmsa.so not found at {path}; build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.msa_version.restype = i32
    lib.msa_last_error_string.restype = ctypes.c_char_p
    lib.msa_landmark_pool.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i32, vp]
    lib.msa_landmark_pool.restype = i32
    lib.msa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, f32,
                                 i32, i32, vp]
    lib.msa_attn_fwd.restype = i32
    lib.msa_attn_fwd_band.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i64, f32,
                                      i32, i32, vp]
    lib.msa_attn_fwd_band.restype = i32
    lib.msa_attn_fwd_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32, i32,
                                      i64, i32, f32, i32, i32, vp]
    lib.msa_attn_fwd_rows.restype = i32
    lib.msa_attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, f32, i32,
                                      i32, i64, vp, ctypes.c_size_t, vp, vp, vp]
    lib.msa_attn_fwd_host.restype = i32
    lib.msa_attn_fwd_host_workspace_size.argtypes = [i64, i32, i32, i32, i32, i64, i32, i32]
    lib.msa_attn_fwd_host_workspace_size.restype = ctypes.c_size_t
    lib.msa_block_select.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, i32, i32, vp]
    lib.msa_block_select.restype = i32
    lib.msa_attn_fwd_select.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32,
                                        i32, f32, i32, i32, vp]
    lib.msa_attn_fwd_select.restype = i32
    lib.msa_attn_fwd_topk_workspace_size.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.msa_attn_fwd_topk_workspace_size.restype = ctypes.c_size_t
    lib.msa_attn_fwd_topk.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32, i32, f32,
                                      i32, i32, vp, ctypes.c_size_t, vp]
    lib.msa_attn_fwd_topk.restype = i32
    lib.msa_attn_fwd_topk_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32,
                                              i32, f32, i32, i32, vp]
    lib.msa_attn_fwd_topk_noalloc.restype = i32
    lib.msa_attn_fwd_global_rows.argtypes = [vp, vp, vp, vp, i64, vp, vp, i64, i32, i32, i32, f32,
                                             i32, i32, vp, ctypes.c_size_t, vp]
    lib.msa_attn_fwd_global_rows.restype = i32
    lib.msa_attn_fwd_global_rows_workspace_size.argtypes = [i64, i64, i32, i32, i32]
    lib.msa_attn_fwd_global_rows_workspace_size.restype = ctypes.c_size_t
    lib.msa_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32,
                                 i64, i32, f32, i32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.msa_attn_bwd.restype = i32
    lib.msa_attn_bwd_workspace_size.argtypes = [i64, i32, i32, i32, i32]
    lib.msa_attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.msa_attn_bwd_global_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp, vp,
                                             i64, i32, i32, i32, i64, i32, f32, i32, i32, i32,
                                             vp, ctypes.c_size_t, vp]
    lib.msa_attn_bwd_global_rows.restype = i32
    lib.msa_attn_bwd_global_rows_workspace_size.argtypes = [i64, i64, i32, i32, i32, i32]
    lib.msa_attn_bwd_global_rows_workspace_size.restype = ctypes.c_size_t
    lib.msa_attn_fwd_partial.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32, i32,
                                         i64, f32, i32, vp]
    lib.msa_attn_fwd_partial.restype = i32
    lib.msa_attn_fwd_partial_merge.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, i32,
                                               i32, i64, f32, i32, vp]
    lib.msa_attn_fwd_partial_merge.restype = i32
    lib.msa_lse_merge.argtypes = [vp, vp, i32, vp, vp, i64, i32, i32, i32, vp]
    lib.msa_lse_merge.restype = i32
    lib.msa_attn_uses_tensor_cores.argtypes = [i32, i32, i32, i32]
    lib.msa_attn_uses_tensor_cores.restype = i32
    lib.msa_attn_fwd_topk_uses_tensor_cores.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.msa_attn_fwd_topk_uses_tensor_cores.restype = i32
    lib.msa_device_status.argtypes = [i32]
    lib.msa_device_status.restype = i32
    lib.msa_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.msa_debug_set_wait_limit_ns.restype = None
    lib.msa_debug_force_single_cta.argtypes = [i32]
    lib.msa_debug_force_single_cta.restype = None
    lib.msa_debug_set_max_clusters.argtypes = [i32]
    lib.msa_debug_set_max_clusters.restype = None
    lib.msa_debug_bounds_build.argtypes = []
    lib.msa_debug_bounds_build.restype = i32
    return lib


_lib = load_library()
if DEBUG_BOUNDS and _lib.msa_debug_bounds_build() != 1:
    raise ImportError(f"{LIB_PATH} is not the bounds-checked build")


def debug_bounds_build() -> bool:
    """True when the loaded library is the bounds-checked build."""
    return bool(_lib.msa_debug_bounds_build())


def _check(status: int) -> None:
    if status != MSA_OK:
        raise MsaError(status, _lib.msa_last_error_string().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MSA_F32
    if t.dtype == torch.bfloat16:
        return MSA_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def version() -> int:
    return int(_lib.msa_version())


def uses_tensor_cores(Hq: int, Hkv: int, d: int, dtype: torch.dtype) -> bool:
    return bool(_lib.msa_attn_uses_tensor_cores(Hq, Hkv, d, MSA_BF16 if dtype == torch.bfloat16
                                                else MSA_F32))


def topk_uses_tensor_cores(n: int, Hq: int, Hkv: int, d: int, n_landmarks: int,
                           dtype: torch.dtype) -> bool:
    return bool(_lib.msa_attn_fwd_topk_uses_tensor_cores(
        n, Hq, Hkv, d, n_landmarks, MSA_BF16 if dtype == torch.bfloat16 else MSA_F32))


def device_status(clear: bool = True) -> int:
    return int(_lib.msa_device_status(1 if clear else 0))


def set_wait_limit_ns(ns: int) -> None:
    _lib.msa_debug_set_wait_limit_ns(int(ns))


def force_single_cta(on: bool) -> None:
    """Test hook: run the single-CTA tensor-core attention kernel where the
    CTA-pair kernel would run (msa_debug_force_single_cta)."""
    _lib.msa_debug_force_single_cta(1 if on else 0)


def set_max_clusters(n: int) -> None:
    """Test hook: run the persistent CTA-pair kernels on at most n pairs
    (0: as many as fit) (msa_debug_set_max_clusters)."""
    _lib.msa_debug_set_max_clusters(int(n))


def landmark_pool(k: torch.Tensor, v: torch.Tensor, k_lm: torch.Tensor, v_lm: torch.Tensor,
                  stream=None) -> None:
    """msa_landmark_pool: block means of k, v [n, Hkv, d] into k_lm, v_lm [G, Hkv, d]."""
    n, Hkv, d = k.shape
    G = k_lm.shape[0]
    _check(_lib.msa_landmark_pool(_ptr(k), _ptr(v), _ptr(k_lm), _ptr(v_lm), n, Hkv, d, G, _dt(k),
                                  _stream(stream)))


def attn_fwd(q, k, v, k_lm, v_lm, out, lse, window: int, n_landmarks: int, scale: float,
             stream=None) -> None:
    """msa_attn_fwd: window + landmark attention; out [n, Hq, d], lse [Hq, n] fp32."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(k_lm), _ptr(v_lm), _ptr(out),
                             _ptr(lse), n, Hq, Hkv, d, int(window), int(n_landmarks),
                             float(scale), _dt(q), _dt(out), _stream(stream)))


def attn_fwd_band(q, k, v, out, lse, band_block: int, band_half: int, scale: float,
                  stream=None) -> None:
    """msa_attn_fwd_band: block-band attention (not causal)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_fwd_band(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), n, Hq, Hkv, d,
                                  int(band_block), int(band_half), float(scale), _dt(q), _dt(out),
                                  _stream(stream)))


def attn_fwd_rows(q_rows, k, v, k_lm, v_lm, out_rows, lse, q_start: int, window: int,
                  n_landmarks: int, scale: float, stream=None) -> None:
    """msa_attn_fwd_rows: query rows [q_start, q_start + len(q_rows)) of the
    window + landmark attention; lse is the full [Hq, n] array (its columns
    q_start.. are written)."""
    n_q, Hq, d = q_rows.shape
    n, Hkv, _ = k.shape
    if lse.shape != (Hq, n) or not lse.is_contiguous():
        raise ValueError("lse must be the contiguous [Hq, n] array")
    lse_ptr = lse.data_ptr() + 4 * int(q_start)
    _check(_lib.msa_attn_fwd_rows(_ptr(q_rows), _ptr(k), _ptr(v), _ptr(k_lm), _ptr(v_lm),
                                  _ptr(out_rows), ctypes.c_void_p(lse_ptr), n, int(q_start), n_q,
                                  n, Hq, Hkv, d, int(window), int(n_landmarks), float(scale),
                                  _dt(q_rows), _dt(out_rows), _stream(stream)))


def host_workspace_size(n: int, Hq: int, Hkv: int, d: int, n_landmarks: int, chunk_rows: int,
                        in_dtype: torch.dtype, out_dtype: torch.dtype) -> int:
    """msa_attn_fwd_host_workspace_size (bytes of device workspace)."""
    ws = int(_lib.msa_attn_fwd_host_workspace_size(
        n, Hq, Hkv, d, n_landmarks, int(chunk_rows),
        MSA_BF16 if in_dtype == torch.bfloat16 else MSA_F32,
        MSA_BF16 if out_dtype == torch.bfloat16 else MSA_F32))
    if ws == 0:
        raise MsaError(MSA_ERR_INVALID_ARG, "invalid sizes for msa_attn_fwd_host")
    return ws


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("msa_attn_fwd_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd_host(hq, hk, hv, hout, hlse, window: int, n_landmarks: int, scale: float,
                  chunk_rows: int, workspace: torch.Tensor, stream=None, copy_in=None,
                  copy_out=None) -> None:
    """msa_attn_fwd_host: host q [n, Hq, d], k, v [n, Hkv, d] -> host out
    [n, Hq, d], lse [Hq, n], streamed through the device workspace; returns
    with the results final."""
    n, Hq, d = hq.shape
    Hkv = hk.shape[1]
    _check(_lib.msa_attn_fwd_host(
        _host_ptr(hq), _host_ptr(hk), _host_ptr(hv), _host_ptr(hout), _host_ptr(hlse), n, Hq, Hkv,
        d, int(window), int(n_landmarks), float(scale), _dt(hq), _dt(hout), int(chunk_rows),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
        None if copy_in is None else ctypes.c_void_p(copy_in.cuda_stream),
        None if copy_out is None else ctypes.c_void_p(copy_out.cuda_stream)))


def block_select(q, k_lm, sel, cnt, window: int, top_k: int, stream=None) -> None:
    """msa_block_select: top-k key blocks per 128-row query block and KV group."""
    n, Hq, d = q.shape
    G, Hkv, _ = k_lm.shape
    _check(_lib.msa_block_select(_ptr(q), _ptr(k_lm), _ptr(sel), _ptr(cnt), n, Hq, Hkv, d,
                                 int(window), G, int(top_k), _dt(q), _stream(stream)))


def attn_fwd_select(q, k, v, sel, cnt, out, lse, window: int, n_landmarks: int, top_k: int,
                    scale: float, stream=None) -> None:
    """msa_attn_fwd_select: window + the selected key blocks."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_fwd_select(_ptr(q), _ptr(k), _ptr(v), _ptr(sel), _ptr(cnt), _ptr(out),
                                    _ptr(lse), n, Hq, Hkv, d, int(window), int(n_landmarks),
                                    int(top_k), float(scale), _dt(q), _dt(out), _stream(stream)))


def topk_workspace_size(n: int, Hkv: int, d: int, n_landmarks: int, top_k: int,
                        dtype: torch.dtype) -> int:
    return int(_lib.msa_attn_fwd_topk_workspace_size(n, Hkv, d, n_landmarks, top_k,
                                                     MSA_BF16 if dtype == torch.bfloat16
                                                     else MSA_F32))


def attn_fwd_topk(q, k, v, out, lse, window: int, n_landmarks: int, top_k: int, scale: float,
                  workspace: torch.Tensor, stream=None) -> None:
    """msa_attn_fwd_topk: pool, select and attend in one call (workspace given)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_fwd_topk(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), n, Hq, Hkv, d,
                                  int(window), int(n_landmarks), int(top_k), float(scale), _dt(q),
                                  _dt(out), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_fwd_topk_noalloc(q, k, v, out, lse, window: int, n_landmarks: int, top_k: int,
                          scale: float, stream=None) -> None:
    """msa_attn_fwd_topk_noalloc: the one-call top-k path on the library's
    fixed per-device scratch (no workspace argument)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_fwd_topk_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), n, Hq,
                                          Hkv, d, int(window), int(n_landmarks), int(top_k),
                                          float(scale), _dt(q), _dt(out), _stream(stream)))


def global_rows_workspace_size(n: int, n_global: int, Hq: int, Hkv: int, d: int) -> int:
    return int(_lib.msa_attn_fwd_global_rows_workspace_size(n, n_global, Hq, Hkv, d))


def attn_fwd_global_rows(q, k, v, rows, out, lse, scale: float, workspace: torch.Tensor,
                         stream=None) -> None:
    """msa_attn_fwd_global_rows: rows (int64 positions on the device) attend
    every key j <= their position; their rows of out / lse are overwritten."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    if rows.dtype != torch.int64:
        raise TypeError("rows must be int64")
    _check(_lib.msa_attn_fwd_global_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), rows.numel(),
                                         _ptr(out), _ptr(lse), n, Hq, Hkv, d, float(scale),
                                         _dt(q), _dt(out), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def attn_bwd_workspace_size(n: int, Hq: int, Hkv: int, d: int, n_landmarks: int) -> int:
    return int(_lib.msa_attn_bwd_workspace_size(n, Hq, Hkv, d, n_landmarks))


def attn_bwd(q, k, v, k_lm, v_lm, out, lse, dout, dq, dk, dv, window: int, n_landmarks: int,
             scale: float, workspace: torch.Tensor, stream=None) -> None:
    """msa_attn_bwd: dq, dk, dv of sum <dout, out> (landmark gradients
    scattered to their tokens)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    _check(_lib.msa_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(k_lm), _ptr(v_lm), _ptr(out),
                             _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), n, Hq, Hkv, d,
                             int(window), int(n_landmarks), float(scale), _dt(q), _dt(out),
                             _dt(dq), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_bwd_global_rows_workspace_size(n: int, n_global: int, Hq: int, Hkv: int, d: int,
                                        n_landmarks: int) -> int:
    return int(_lib.msa_attn_bwd_global_rows_workspace_size(n, n_global, Hq, Hkv, d,
                                                            n_landmarks))


def attn_bwd_global_rows(q, k, v, k_lm, v_lm, out, lse, dout, rows, dq, dk, dv, window: int,
                         n_landmarks: int, scale: float, workspace: torch.Tensor,
                         stream=None) -> None:
    """msa_attn_bwd_global_rows: gradients of the compression-token pattern
    (window + landmarks, then the global rows)."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    if rows.dtype != torch.int64:
        raise TypeError("rows must be int64")
    _check(_lib.msa_attn_bwd_global_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(k_lm), _ptr(v_lm), _ptr(out), _ptr(lse), _ptr(dout),
        _ptr(rows), rows.numel(), _ptr(dq), _ptr(dk), _ptr(dv), n, Hq, Hkv, d, int(window),
        int(n_landmarks), float(scale), _dt(q), _dt(out), _dt(dq), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def attn_fwd_partial(q, k_chunk, v_chunk, out_part, lse_part, q_start: int, kv_start: int,
                     window: int, scale: float, stream=None) -> None:
    """msa_attn_fwd_partial: one Ring Attention round's partial (fp32 out_part)."""
    n_q, Hq, d = q.shape
    n_kv, Hkv, _ = k_chunk.shape
    _check(_lib.msa_attn_fwd_partial(_ptr(q), _ptr(k_chunk), _ptr(v_chunk), _ptr(out_part),
                                     _ptr(lse_part), n_q, int(q_start), n_kv, int(kv_start), Hq,
                                     Hkv, d, int(window), float(scale), _dt(q), _stream(stream)))


def attn_fwd_partial_merge(q, k_chunk, v_chunk, out_run, lse_run, q_start: int, kv_start: int,
                           window: int, scale: float, stream=None) -> None:
    """msa_attn_fwd_partial_merge: one ring round merged into (out_run, lse_run) in place."""
    n_q, Hq, d = q.shape
    n_kv, Hkv, _ = k_chunk.shape
    _check(_lib.msa_attn_fwd_partial_merge(_ptr(q), _ptr(k_chunk), _ptr(v_chunk), _ptr(out_run),
                                           _ptr(lse_run), n_q, int(q_start), n_kv, int(kv_start),
                                           Hq, Hkv, d, int(window), float(scale), _dt(q),
                                           _stream(stream)))


def lse_merge(o_parts, lse_parts, out, lse, stream=None) -> None:
    """msa_lse_merge: exact LSE-weighted merge of partials (lists of tensors)."""
    P = len(o_parts)
    if P != len(lse_parts):
        raise ValueError("o_parts and lse_parts differ in length")
    n, Hq, d = out.shape
    arr_o = (ctypes.c_void_p * max(P, 1))(*[t.data_ptr() for t in o_parts])
    arr_l = (ctypes.c_void_p * max(P, 1))(*[t.data_ptr() for t in lse_parts])
    for t in list(o_parts) + list(lse_parts):
        _ptr(t)
    _check(_lib.msa_lse_merge(arr_o, arr_l, P, _ptr(out), _ptr(lse), n, Hq, d, _dt(out),
                              _stream(stream)))
