import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


# XS_TEST_LIBRARY=debug runs the GPU tests on the debug library (the same
# kernels with in-kernel bounds checks on every computed global-memory index,
# built by build.build(debug_bounds=True)) instead of the release one, and
# requires after every GPU test that no check failed on the device.
DEBUG_LIBRARY = os.environ.get("XS_TEST_LIBRARY") == "debug"


@pytest.fixture(autouse=True)
def _library_under_test(request):
    if not DEBUG_LIBRARY or request.node.get_closest_marker("gpu") is None:
        yield
        return
    from paged_kv_cache_xs_gb300 import build as xsbuild
    from paged_kv_cache_xs_gb300 import ops
    xsbuild.build(debug_bounds=True)
    lib = ops.load_debug()
    prev = ops.use_library(lib)
    try:
        yield
        failures = ops.xs_debug_bounds_failures(reset=True, lib=lib)
        assert failures == 0, f"{failures} in-kernel bounds checks failed"
    finally:
        ops.use_library(prev)
