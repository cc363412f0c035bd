"""Memory-safety evidence without a sanitizer: the small GPU parity grid run
against the bounds-checked build of the library.

libmsa_debug.so is compiled with -DMSA_DEBUG_BOUNDS: every kernel tests
each computed global offset against the extent its entry point's contract
gives that buffer, and each TMA box origin against its tensor; a failure
records MSA_ERR_INVALID_ARG in the device status word and prints its
source line (nothing traps).  This test builds that library and runs every
GPU test except the full-size ones (marker ``large``) and the timeout
tests in a child pytest with MSA_DEBUG_BOUNDS=1, where conftest checks
after each test that the status word is clear and that the canary guard
bytes around every output and workspace buffer are intact.  The child
must pass and must print no range-check failure."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu

CHILD_FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_pair_kernel.py",
               "tests/test_gpu_rows.py", "tests/test_gpu_topk.py", "tests/test_gpu_compressed.py",
               "tests/test_gpu_bwd.py", "tests/test_zz_no_alloc.py"]


@pytest.mark.large
def test_small_parity_grid_under_range_checks():
    if os.environ.get("MSA_DEBUG_BOUNDS") == "1":
        pytest.skip("already running against the bounds-checked build")
    from long_context_sparse_landmark_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, MSA_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           "-m", "gpu and not large", *CHILD_FILES]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    out = r.stdout + r.stderr
    print(out[-3000:])
    assert r.returncode == 0, out[-3000:]
    assert "msa bounds check" not in out, "a range check failed"
    assert " passed" in out
