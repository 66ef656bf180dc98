"""The failure path of the bounded device waits, on a GPU, without faulting it.

Every mbarrier wait in the GEMM pipelines is bounded: when it runs out the kernel records a
code in the device status word and returns instead of hanging or trapping. The self-test
kernel waits, with that same wait, on a barrier nothing arrives at; the host must then read
MX_ERR_DEVICE_TIMEOUT, clear it, and find the context still usable.
"""
import time

import numpy as np
import pytest

import oracle
from gpu_util import bf16_host, dev, native

pytestmark = pytest.mark.gpu

MX_ERR_DEVICE_TIMEOUT = 6


@pytest.fixture(scope="module")
def mx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m = native()
    assert m.device_status(clear=True) == 0
    yield m
    assert m.device_status(clear=True) == 0


def test_bounded_wait_times_out_reports_and_the_context_survives(mx):
    import torch
    t0 = time.perf_counter()
    mx.selftest_wait_timeout()
    st = mx.device_status(clear=True)                 # synchronises
    dt = time.perf_counter() - t0
    assert st == MX_ERR_DEVICE_TIMEOUT, mx.status_string(st)
    assert 1.0 < dt < 60.0, f"the wait took {dt:.2f} s"
    assert mx.device_status(clear=True) == 0          # cleared
    # the context still runs kernels correctly
    rng = np.random.default_rng(91)
    codes = rng.integers(0, 256, size=(64, 128), dtype=np.uint8)
    sf = rng.integers(118, 125, size=(64, 8), dtype=np.uint8)
    out = torch.empty((64, 256), dtype=torch.bfloat16, device="cuda")
    mx.mxfp4_dequant(dev(codes), dev(sf), out)
    np.testing.assert_array_equal(bf16_host(out), oracle.mxfp4_dequant(codes, sf))
    assert mx.device_status(clear=True) == 0
