import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def root():
    return ROOT


@pytest.fixture(autouse=True)
def _no_bounds_violations():
    """Under the bounds-checked build (MOE_EXPECT_DEBUG set by
    test_gpu_debug_bounds), every test must leave the violation count at 0."""
    yield
    if os.environ.get("MOE_EXPECT_DEBUG"):
        from expert_cache_serving_gb300 import moecache as mc

        assert mc.lib.moe_debug_bounds_enabled() == 1, "MOECACHE_LIB is not the bounds-checked build"
        count, site = mc.moe_debug_violations()
        assert count == 0, f"{count} bounds violations, first at check site {site}"
