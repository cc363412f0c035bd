"""fp64 CPU oracle for window + landmark sparse attention (test infrastructure).

This package is the correctness authority the CUDA library is checked
against.  It is TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke``
and the benchmark's CPU-baseline leg may import it.  It shares no code with
the CUDA path and never imports it.

The arithmetic lives in ``msa_oracle.c`` (plain C, fp64, OpenMP over rows and
heads); this module compiles it with gcc on first use and marshals numpy
arrays into it.  The definition it follows, and the reading of the pages it
takes, is stated at the top of ``msa_oracle.c``.

Inputs are numpy arrays: ``float32``, or ``uint16`` holding bf16 bit patterns
(``dtype="bf16"``).  Outputs are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the C oracle into ``libmsa_oracle.so`` (gcc, fp64, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_landmark_pool.argtypes = [vp, i32, i64, i32, i32, i32, vp]
    lib.oracle_landmark_pool.restype = i32
    lib.oracle_attn_rows.argtypes = [vp, vp, i64, vp, vp, i64, i64, i32,
                                     i32, i32, i32, i64, vp, vp, i32, i64,
                                     dbl, vp, vp]
    lib.oracle_attn_rows.restype = i32
    lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, i64, i32, dbl,
                                    vp, vp, vp]
    lib.oracle_attn_bwd.restype = i32
    lib.oracle_attn_bwd_dq_rows.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, i64, i32,
                                            dbl, vp, i64, vp]
    lib.oracle_attn_bwd_dq_rows.restype = i32
    lib.oracle_attn_bwd_dkdv_keys.argtypes = [vp, vp, vp, vp, i32, i64, i32, i32, i32, i64, i32,
                                              dbl, vp, vp, i64, vp, vp]
    lib.oracle_attn_bwd_dkdv_keys.restype = i32
    lib.oracle_attn_band_rows.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32,
                                          i32, i32, i64, i64, dbl, vp, vp]
    lib.oracle_attn_band_rows.restype = i32
    lib.oracle_block_scores.argtypes = [vp, i32, i64, i32, i32, i32, vp, i32, i64,
                                        i64, i64, vp]
    lib.oracle_block_scores.restype = i32
    lib.oracle_attn_select_rows.argtypes = [vp, vp, i64, vp, vp, i64, i32, i32, i32,
                                            i32, i64, i64, i64, vp, vp, i32, dbl, vp,
                                            vp]
    lib.oracle_attn_select_rows.restype = i32
    lib.oracle_lse_merge.argtypes = [vp, vp, i32, i64, i32, i32, vp, vp]
    lib.oracle_lse_merge.restype = i32
    lib.oracle_set_threads.argtypes = [i32]
    lib.oracle_get_threads.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _configure(ctypes.CDLL(build()))
        return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle inputs must be float32 or uint16 (bf16 bits), got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def landmark_pool(x: np.ndarray, n_landmarks: int) -> np.ndarray:
    """Block means of x [n, H, d] over G = n_landmarks blocks -> [G, H, d] fp64."""
    x = np.ascontiguousarray(x)
    n, H, d = x.shape
    out = np.empty((n_landmarks, H, d), dtype=np.float64)
    rc = _load().oracle_landmark_pool(_ptr(x), _dtype_code(x), n, H, d,
                                      n_landmarks, _ptr(out))
    if rc != 0:
        raise ValueError("landmark_pool: n must be a positive multiple of G")
    return out


def attn(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int,
         n_landmarks: int, scale: float, rows=None, q_start: int = 0,
         kv_start: int = 0, q_positions=None, landmarks=None):
    """Window + landmark attention in fp64.

    q: [n_q, Hq, d] query rows at global positions q_start + index; k, v:
    [n_kv, Hkv, d] at global positions kv_start + index.  ``rows`` selects a
    subset of q's rows (indices into q).  Alternatively ``q_positions`` gives
    the global position of every row of q (q then holds exactly those rows,
    e.g. a gathered sample).  Landmarks (G = n_landmarks > 0) are the block
    means of k and v over the whole sequence, which requires kv_start == 0;
    ``landmarks=(k_lm, v_lm)`` passes ones already computed by
    ``landmark_pool`` for these k, v.
    Returns (O [n_rows, Hq, d], lse [Hq, n_rows]).
    """
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    dt = _dtype_code(q)
    if _dtype_code(k) != dt or _dtype_code(v) != dt:
        raise TypeError("q, k, v must share one dtype")
    n_q, Hq, d = q.shape
    n_kv, Hkv, _ = k.shape
    if q_positions is not None:
        if rows is not None:
            raise ValueError("give rows or q_positions, not both")
        pos = np.ascontiguousarray(np.asarray(q_positions, dtype=np.int64))
        if len(pos) != n_q:
            raise ValueError("q_positions must have one entry per row of q")
        qg = q
    else:
        if rows is None:
            rows = np.arange(n_q, dtype=np.int64)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        qg = np.ascontiguousarray(q[rows])
        pos = np.ascontiguousarray(rows + int(q_start), dtype=np.int64)
    n_rows = len(pos)
    G = int(n_landmarks)
    if G > 0:
        if kv_start != 0:
            raise ValueError("landmarks need the whole sequence (kv_start == 0)")
        if landmarks is None:
            k_lm = landmark_pool(k, G)
            v_lm = landmark_pool(v, G)
        else:
            k_lm = np.ascontiguousarray(landmarks[0], dtype=np.float64)
            v_lm = np.ascontiguousarray(landmarks[1], dtype=np.float64)
            if k_lm.shape != (G, Hkv, d) or v_lm.shape != (G, Hkv, d):
                raise ValueError("landmarks must be [G, Hkv, d]")
        B = n_kv // G
        lm_k, lm_v = _ptr(k_lm), _ptr(v_lm)
    else:
        B = 1
        lm_k = lm_v = None
    out = np.empty((n_rows, Hq, d), dtype=np.float64)
    lse = np.empty((Hq, n_rows), dtype=np.float64)
    rc = _load().oracle_attn_rows(_ptr(qg), _ptr(pos), n_rows, _ptr(k),
                                  _ptr(v), n_kv, int(kv_start), dt, Hq, Hkv, d,
                                  int(window), lm_k, lm_v, G, B, float(scale),
                                  _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("attn: inconsistent arguments")
    return out, lse


def attn_band(q: np.ndarray, k: np.ndarray, v: np.ndarray, band_block: int,
              band_half: int, scale: float, rows=None, q_positions=None):
    """Block-band attention in fp64: row i attends every key of the blocks
    (size band_block) within band_half blocks of its own, not causal.
    Returns (O [n_rows, Hq, d], lse [Hq, n_rows])."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    dt = _dtype_code(q)
    if _dtype_code(k) != dt or _dtype_code(v) != dt:
        raise TypeError("q, k, v must share one dtype")
    n_q, Hq, d = q.shape
    n_kv, Hkv, _ = k.shape
    if q_positions is not None:
        pos = np.ascontiguousarray(np.asarray(q_positions, dtype=np.int64))
        qg = q
    else:
        rows = np.arange(n_q, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
        qg = np.ascontiguousarray(q[rows])
        pos = np.ascontiguousarray(rows)
    out = np.empty((len(pos), Hq, d), dtype=np.float64)
    lse = np.empty((Hq, len(pos)), dtype=np.float64)
    rc = _load().oracle_attn_band_rows(_ptr(qg), _ptr(pos), len(pos), _ptr(k), _ptr(v), n_kv,
                                       dt, Hq, Hkv, d, int(band_block), int(band_half),
                                       float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("attn_band: inconsistent arguments")
    return out, lse


def block_scores(q: np.ndarray, k: np.ndarray, n_landmarks: int, window: int,
                 q_block: int = 128) -> np.ndarray:
    """Scores [n_qb, Hkv, G] (fp64) of every key block for every query
    block and KV group; -inf where the block is not wholly before the
    window of the query block's first row."""
    q = np.ascontiguousarray(q)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = int(n_landmarks)
    k_lm = landmark_pool(k, G)
    n_qb = (n + q_block - 1) // q_block
    scores = np.empty((n_qb, Hkv, G), dtype=np.float64)
    rc = _load().oracle_block_scores(_ptr(q), _dtype_code(q), n, Hq, Hkv, d, _ptr(k_lm), G,
                                     n // G, int(window), int(q_block), _ptr(scores))
    if rc != 0:
        raise ValueError("block_scores: inconsistent arguments")
    return scores


def select_top_k(scores: np.ndarray, top_k: int):
    """The top-k blocks of every (query block, KV group): highest scores
    first, ties to the lower block index, -inf never chosen.  Returns
    (sel [n_qb, Hkv, top_k] int32 in ascending block order, cnt [n_qb, Hkv])."""
    n_qb, Hkv, G = scores.shape
    sel = np.zeros((n_qb, Hkv, max(top_k, 1)), dtype=np.int32)
    cnt = np.zeros((n_qb, Hkv), dtype=np.int32)
    for t in range(n_qb):
        for c in range(Hkv):
            cand = [l for l in range(G) if np.isfinite(scores[t, c, l])]
            cand.sort(key=lambda l: (-scores[t, c, l], l))
            chosen = sorted(cand[:top_k])
            cnt[t, c] = len(chosen)
            sel[t, c, :len(chosen)] = chosen
    return sel[:, :, :top_k] if top_k > 0 else sel[:, :, :0], cnt


def attn_select(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int, n_landmarks: int,
                sel: np.ndarray, cnt: np.ndarray, scale: float, q_block: int = 128,
                rows=None, q_positions=None):
    """Attention over each row's causal window plus every token of its query
    block's selected key blocks (sel/cnt as select_top_k returns).  Returns
    (O [n_rows, Hq, d], lse [Hq, n_rows]) in fp64."""
    q = np.ascontiguousarray(q)
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    dt = _dtype_code(q)
    n_q, Hq, d = q.shape
    n, Hkv, _ = k.shape
    if q_positions is not None:
        pos = np.ascontiguousarray(np.asarray(q_positions, dtype=np.int64))
        qg = q
    else:
        rows = np.arange(n_q, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
        qg = np.ascontiguousarray(q[rows])
        pos = np.ascontiguousarray(rows)
    top_k = sel.shape[2]
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    cnt = np.ascontiguousarray(cnt, dtype=np.int32)
    out = np.empty((len(pos), Hq, d), dtype=np.float64)
    lse = np.empty((Hq, len(pos)), dtype=np.float64)
    rc = _load().oracle_attn_select_rows(_ptr(qg), _ptr(pos), len(pos), _ptr(k), _ptr(v), n, dt,
                                         Hq, Hkv, d, int(window), n // int(n_landmarks),
                                         int(q_block), _ptr(sel), _ptr(cnt), int(top_k),
                                         float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("attn_select: inconsistent arguments")
    return out, lse


def attn_compressed(q: np.ndarray, k: np.ndarray, v: np.ndarray, window: int, block: int,
                    global_rows, scale: float, rows=None, q_positions=None):
    """Compression tokens plus global query rows, after the Block-Sparse
    Flash Attention paragraph of "Training at 1M+ Token Context: Ring
    Attention, YaRN, NTK-Aware Scaling GPU Cost" (local rows see a sliding
    window, compression tokens summarise distant context, global tokens
    attend to everything; 256 compression tokens per 8192-token chunk).

    A compression token is the mean of K (and of V) over one ``block``-token
    sub-block (block = 32 gives 256 per 8192 tokens).  A row not in
    ``global_rows`` attends its window and the compression tokens of the
    sub-blocks wholly before it -- window + landmark attention with
    G = n / block.  A row in ``global_rows`` attends every key j <= i and
    nothing else.  Returns (O [n_rows, Hq, d], lse [Hq, n_rows]) for
    ``rows`` (indices of q, default all), or, with ``q_positions``, for the
    rows q holds, at those positions.
    """
    n = k.shape[0]
    if block < 1 or n % block != 0:
        raise ValueError("block must divide n")
    if q_positions is not None:
        pos = np.asarray(q_positions, dtype=np.int64)
        qg = np.ascontiguousarray(q)
    else:
        pos = np.arange(n, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
        qg = np.ascontiguousarray(q[pos])
    is_global = np.isin(pos, np.asarray(global_rows, dtype=np.int64))
    Hq, d = q.shape[1], q.shape[2]
    out = np.empty((len(pos), Hq, d), dtype=np.float64)
    lse = np.empty((Hq, len(pos)), dtype=np.float64)
    local = np.nonzero(~is_global)[0]
    glob = np.nonzero(is_global)[0]
    if local.size:
        out[local], lse[:, local] = attn(qg[local], k, v, window, n // block, scale,
                                         q_positions=pos[local])
    if glob.size:
        out[glob], lse[:, glob] = attn(qg[glob], k, v, n, 0, scale, q_positions=pos[glob])
    return out, lse


def attn_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, window: int,
             n_landmarks: int, scale: float):
    """Gradients (dQ [n,Hq,d], dK, dV [n,Hkv,d], fp64) of sum <dout, O> for
    window + landmark attention over the whole sequence, landmark gradients
    scattered back to the tokens they average (1/B each)."""
    q, k, v, dout = (np.ascontiguousarray(x) for x in (q, k, v, dout))
    dt = _dtype_code(q)
    if any(_dtype_code(x) != dt for x in (k, v, dout)):
        raise TypeError("q, k, v, dout must share one dtype")
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    dq = np.empty((n, Hq, d), dtype=np.float64)
    dk = np.empty((n, Hkv, d), dtype=np.float64)
    dv = np.empty((n, Hkv, d), dtype=np.float64)
    rc = _load().oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), dt, n, Hq, Hkv, d,
                                 int(window), int(n_landmarks), float(scale), _ptr(dq),
                                 _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("attn_bwd: inconsistent arguments")
    return dq, dk, dv


def attn_bwd_dq_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray, window: int,
                     n_landmarks: int, scale: float, rows):
    """dQ [n_rows, Hq, d] (fp64) of the listed rows only (q, dout whole)."""
    q, k, v, dout = (np.ascontiguousarray(x) for x in (q, k, v, dout))
    dt = _dtype_code(q)
    n, Hq, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.empty((len(rows), Hq, d), dtype=np.float64)
    rc = _load().oracle_attn_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), dt, n, Hq,
                                         k.shape[1], d, int(window), int(n_landmarks),
                                         float(scale), _ptr(rows), len(rows), _ptr(dq))
    if rc != 0:
        raise ValueError("attn_bwd_dq_rows: inconsistent arguments")
    return dq


def attn_bwd_dkdv_keys(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                       window: int, n_landmarks: int, scale: float, keys, kv_heads):
    """dK, dV [n_keys, d] (fp64) of the listed (key position, KV head) pairs
    only, for window + landmark attention over the whole sequence (q, k, v,
    dout whole): the window rows of each key plus its block's landmark
    gradient divided by the block size; row statistics are computed only
    for the rows that see a listed key or its landmark."""
    q, k, v, dout = (np.ascontiguousarray(x) for x in (q, k, v, dout))
    dt = _dtype_code(q)
    if any(_dtype_code(x) != dt for x in (k, v, dout)):
        raise TypeError("q, k, v, dout must share one dtype")
    n, Hq, d = q.shape
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    kv_heads = np.ascontiguousarray(np.asarray(kv_heads, dtype=np.int32))
    if keys.shape != kv_heads.shape:
        raise ValueError("one KV head per listed key")
    dk = np.empty((len(keys), d), dtype=np.float64)
    dv = np.empty((len(keys), d), dtype=np.float64)
    rc = _load().oracle_attn_bwd_dkdv_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), dt, n, Hq,
                                           k.shape[1], d, int(window), int(n_landmarks),
                                           float(scale), _ptr(keys), _ptr(kv_heads), len(keys),
                                           _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("attn_bwd_dkdv_keys: inconsistent arguments")
    return dk, dv


def attn_bwd_compressed(q: np.ndarray, k: np.ndarray, v: np.ndarray, dout: np.ndarray,
                        window: int, block: int, global_rows, scale: float):
    """Gradients (dQ, dK, dV, fp64) of sum <dout, O> for the compression-token
    pattern of ``attn_compressed``.  The output of a global row does not
    depend on the window or the compression tokens, and the other rows' do
    not depend on the global rows' queries, so the gradient is the sum of
    the window + compression-token backward with the global rows' dout set
    to zero, and the causal (w = n, no landmarks) backward with only the
    global rows' dout."""
    n = q.shape[0]
    rows = np.asarray(global_rows, dtype=np.int64)
    is_global = np.zeros(n, dtype=bool)
    is_global[rows] = True
    zero = np.zeros_like(dout[:1])
    d_local = np.where(is_global[:, None, None], zero, dout)
    d_glob = np.where(is_global[:, None, None], dout, zero)
    a = attn_bwd(q, k, v, np.ascontiguousarray(d_local), window, n // block, scale)
    if rows.size == 0:
        return a
    b = attn_bwd(q, k, v, np.ascontiguousarray(d_glob), n, 0, scale)
    return tuple(x + y for x, y in zip(a, b))


def lse_merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge P partials: o_parts [P, n, Hq, d], lse_parts [P, Hq, n] (fp64)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    P, n, Hq, d = o_parts.shape
    out = np.empty((n, Hq, d), dtype=np.float64)
    lse = np.empty((Hq, n), dtype=np.float64)
    rc = _load().oracle_lse_merge(_ptr(o_parts), _ptr(lse_parts), P, n, Hq, d,
                                  _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("lse_merge: bad shapes")
    return out, lse


def attended_count(pos: int, window: int, n_landmarks: int, block: int,
                   kv_start: int = 0, n_kv: int | None = None) -> int:
    """Size of row pos's attended set, counted from the set definitions."""
    lo = max(pos - window + 1, kv_start)
    hi = pos if n_kv is None else min(pos, kv_start + n_kv - 1)
    n_win = max(0, hi - lo + 1)
    n_lm = sum(1 for l in range(n_landmarks) if (l + 1) * block <= pos - window + 1)
    return n_win + n_lm
