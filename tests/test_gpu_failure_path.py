"""The failure path of the bounded device waits, on a GPU, without faulting it.

Every mbarrier wait in the GEMM pipelines is bounded: when it runs out the kernel records a
code in the status words (the call's workspace word and the device-wide word) and returns
instead of hanging or trapping. The self-test kernel waits, with that same wait, on a
barrier nothing arrives at; the host must then read MX_ERR_DEVICE_TIMEOUT, clear it, and
find the context still usable. The workspace word is per call and per stream: a forward on
another stream with its own workspace stays clean, and checking it does not wait for the
stream whose wait is running out.
"""
import time

import numpy as np
import pytest

import oracle
from gpu_util import assert_moe_close, bf16_host, dev, native

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


def test_workspace_status_word_is_per_call_and_per_stream(mx):
    import torch
    from workloads import make_config_inputs
    inp = make_config_inputs("tiny")
    x = dev(inp.x).view(torch.bfloat16)
    ids, w = dev(inp.topk_ids), dev(inp.topk_w)
    W = [dev(a) for a in (inp.w13, inp.s13, inp.w2, inp.s2)]
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    ws_a = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(mx.moe_mxfp4_workspace_size(inp.T, inp.H, inp.I, inp.E, inp.K, True), dtype=torch.uint8,
                       device="cuda")
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    ws_b[:16].fill_(0xFF)                               # stale garbage: the forward must clear it
    torch.cuda.synchronize()                            # inputs and fill done before other streams read
    mx.moe_mxfp4_forward(x, ids, w, *W, out, ws_b, stream=s_b)      # warm-up: kernels loaded
    assert mx.check_workspace(ws_b, stream=s_b) == 0
    torch.cuda.synchronize()

    t0 = time.perf_counter()
    mx.selftest_wait_timeout(stream=s_a, workspace=ws_a)            # runs out after ~2 s
    mx.moe_mxfp4_forward(x, ids, w, *W, out, ws_b, stream=s_b)
    st_b = mx.check_workspace(ws_b, stream=s_b)
    t_b = time.perf_counter() - t0
    st_a = mx.check_workspace(ws_a, stream=s_a)
    t_a = time.perf_counter() - t0
    assert st_b == 0, mx.status_string(st_b)
    assert st_a == MX_ERR_DEVICE_TIMEOUT, mx.status_string(st_a)
    assert t_b < 1.0 < t_a, f"check of stream B after {t_b:.2f} s, of stream A after {t_a:.2f} s"
    assert mx.check_workspace(ws_a, stream=s_a) == 0                # cleared by the first check
    assert mx.device_status(clear=True) == MX_ERR_DEVICE_TIMEOUT    # the device-wide word saw it too
    assert mx.device_status(clear=True) == 0
    ref = oracle.moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.w2, inp.s2, inp.I)
    assert_moe_close(bf16_host(out), ref, "forward beside the timed-out wait")
