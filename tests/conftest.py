import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU case")
    config.addinivalue_line("markers", "large: full-size GPU workload (128K tokens and up), "
                                       "left out of the bounds-checked run")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without one fails loudly instead of silently
    # running something else; select with -m "not gpu" on CPU-only hosts.
    pass


@pytest.fixture(autouse=True)
def _canary_guards(request):
    """After every GPU test: no kernel wrote into the guard bytes around the
    test's output and workspace buffers (see gpu_helpers.gempty)."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    from tests import gpu_helpers
    gpu_helpers.check_guards(forget=True)
    if os.environ.get("MSA_DEBUG_BOUNDS") == "1":
        # Under the bounds-checked build no range check may have failed in
        # the test (tests that provoke a status read and clear it themselves).
        from long_context_sparse_landmark_gb300 import _binding
        assert _binding.device_status(clear=True) == 0, "a range check failed"


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle
