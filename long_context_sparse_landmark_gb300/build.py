"""Build libmsa.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel into ``_build/`` and the
objects are linked into ``libmsa.so`` next to this file (CUDA runtime linked
statically, so the library loads on hosts without a GPU driver too).

``build(debug_bounds=True)`` builds the bounds-checked variant instead
(``-DMSA_DEBUG_BOUNDS``, objects in ``_build/debug_bounds/``, library
``libmsa_debug.so``): every kernel range-checks its global offsets and TMA
box origins and records a violation in the device status word.  It is slower
and is only loaded when MSA_DEBUG_BOUNDS=1 is set in the environment.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmsa.so")
LIB_DEBUG = os.path.join(PKG, "libmsa_debug.so")

SOURCES = ["msa_api.cu", "k1_landmark_pool.cu", "k2_attn_simt.cu", "k2_attn_tc.cu",
           "k2_attn_tc2.cu", "k3_lse_merge.cu", "k4_block_select.cu", "k5_global_rows.cu",
           "k6_attn_bwd.cu", "k6_bwd_dq_pair.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmsa")
    return nvcc


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug_bounds: bool = False) -> str:
    """Compile and link libmsa.so (or, with debug_bounds, libmsa_debug.so);
    returns its path.  Skips work when the library is newer than every
    source and header."""
    lib = LIB_DEBUG if debug_bounds else LIB
    out_dir = os.path.join(BUILD, "debug_bounds") if debug_bounds else BUILD
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if debug_bounds:
        extra.append("-DMSA_DEBUG_BOUNDS")

    def compile_one(src):
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
