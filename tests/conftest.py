import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(autouse=True)
def _canary_guard_bands():
    """After every test, the guard bands of the buffers it allocated with
    gpu_util.guarded_empty must be untouched (an out-of-bounds store would show there)."""
    yield
    import gpu_util
    if gpu_util._guarded:
        gpu_util.check_canaries()
