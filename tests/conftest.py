import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _bounds_failures_after_each_test():
    """On the bounds-checked build (RC_BOUNDS_CHECK=1), no cache a test made may
    have failed an index check or a guard, reported by a sync or not."""
    yield
    if os.environ.get("RC_BOUNDS_CHECK") != "1" or "fp8_ring_kv_cache_gb300._binding" not in sys.modules:
        return
    import gc
    gc.collect()  # caches the test dropped are closed (and checked) now
    failures = sys.modules["fp8_ring_kv_cache_gb300._binding"].BOUNDS_FAILURES
    found, failures[:] = list(failures), []
    assert not found, f"bounds-checked build: checks or guards failed in {found}"
