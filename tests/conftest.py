import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session", autouse=True)
def _bounds_checked_run():
    """With ZR_CHECKED_RUN=1 (tests/test_gpu_checked.py runs the parity tests
    that way, against libzr_checked.so): after the session, no bounds check of
    the checked build may have failed."""
    yield
    if os.environ.get("ZR_CHECKED_RUN") != "1":
        return
    from zero_partition_aware_gb300 import zr
    n, code, where = zr.zr_debug_checks()
    assert n == 0, f"the bounds-checked build recorded {n} failed checks (first: check {code} at element {where})"
