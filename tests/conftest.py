"""Shared pytest set-up: the ``gpu`` marker and import paths."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built CUDA library")


@pytest.fixture(autouse=True)
def _bounds_checks_stay_clean(request):
    """Under the bounds-checked library (HICACHE_CHECKED=1), every GPU test
    must leave the device's check words at zero: no kernel decoded a vector
    outside its buffers, the host pool or the run table."""
    yield
    if os.environ.get("HICACHE_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import tiered_kv_cache_gb300 as hc
    assert hc.checked_build(), "HICACHE_CHECKED=1 but the plain library is loaded"
    first, count = hc.check_status(clear=True)
    assert (first, count) == (0, 0), f"failed bounds checks: first {first:#x}, count {count}"
