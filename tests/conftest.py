import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session", autouse=True)
def _libraries_built():
    """Build libmj.so (sm_103a; nvcc cross-compiles without a GPU) and the
    oracle's checker once per session, whichever test runs first: both are
    build products, absent from a fresh checkout."""
    from paged_fp8_kv_gb300.build import build

    import oracle

    build()
    oracle.build()
