"""moe_mxfp4_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers only receive their input and output buffers (a plugin or custom-op interface
whose framework owns every device allocation, or code that must not pay cudaMalloc's
device-wide synchronisation). This entry point runs the same forward on a static scratch
area inside the library instead of a caller workspace. The test calls it through the C
ABI twice in a row, on two different workloads, and checks each output against the
regular entry point (moe_mxfp4_forward with a caller workspace) within the tolerance the
MoE tests use; it also checks that a batch too large for the scratch area is refused.
Collected last on purpose: a run that stops at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import assert_moe_close, bf16_host, dev, native
from workloads import make_moe_inputs

pytestmark = pytest.mark.gpu

MX_ERR_WORKSPACE = 4


@pytest.fixture(scope="module")
def mx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m = native()
    assert m.device_status(clear=True) == 0
    yield m
    assert m.device_status(clear=True) == 0, "a bounded device wait ran out"


def _regular_and_noalloc(mx, inp):
    import torch
    x = dev(inp.x).view(torch.bfloat16)
    routed = inp.topk_ids is not None
    ids = dev(inp.topk_ids) if routed else None
    w = dev(inp.topk_w) if routed else None
    W = [dev(a) for a in (inp.w13, inp.s13, inp.w2, inp.s2)]
    ref_out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(mx.moe_mxfp4_workspace_size(inp.T, inp.H, inp.I, inp.E, inp.K, routed),
                     dtype=torch.uint8, device="cuda")
    mx.moe_mxfp4_forward(x, ids, w, *W, ref_out, ws)

    out = torch.full((inp.T, inp.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    st = mx.lib().moe_mxfp4_forward_noalloc(p(x), p(ids), p(w), p(W[0]), p(W[1]), p(W[2]), p(W[3]), p(out),
                                            inp.T, inp.H, inp.I, inp.E, inp.K, ctypes.c_void_p(stream))
    assert st == 0, mx.status_string(st)
    torch.cuda.synchronize()
    return bf16_host(ref_out), bf16_host(out)


def test_noalloc_matches_regular_forward_twice(mx):
    first = make_moe_inputs(T=96, H=1024, I=512, E=8, K=4, seed=41, routing="uniform")
    second = make_moe_inputs(T=150, H=768, I=384, E=1, K=1, seed=42, routing=None)
    for inp in (first, second):                     # two calls in a row on the shared scratch
        ref, got = _regular_and_noalloc(mx, inp)
        assert_moe_close(got, ref, "noalloc vs regular forward")
        np.testing.assert_array_equal(got, ref)     # same kernels, same order: identical bits


def test_noalloc_refuses_batches_beyond_its_scratch(mx):
    import torch
    T, H, I, E, K = 4096, 7168, 3072, 48, 8
    assert mx.moe_mxfp4_workspace_size(T, H, I, E, K, True) > (32 << 20)
    out = torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda")
    fake = ctypes.c_void_p(out.data_ptr())
    st = mx.lib().moe_mxfp4_forward_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, T, H, I, E, K,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == MX_ERR_WORKSPACE
    assert (out.float() == 0).all()                 # nothing was launched
