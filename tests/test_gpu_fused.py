"""GPU tests of moe_mxfp4_forward_fused, the whole forward as one persistent cooperative
launch ("Current Bug: vLLM produces empty/garbage output": the nvfp4-megamoe-kernel plan,
"Phase 1: CuTeDSL Shared Expert Kernel").

It runs the multi-kernel forward's device code in the same order, so its output must be
bit-identical to moe_mxfp4_forward with tile-layout scales, which the MoE parity tests check
against the oracle step by step. Covered: the tiny config, routing edge cases (dropped ids,
empty experts, several ragged M tiles per expert), ragged K and N tails in both modes, the
full-size shared expert, decode and prefill, two calls in a row on one workspace, CUDA-graph
replay, and the failure path of its grid-wide barrier (a bounded wait that runs out).
"""
import time

import numpy as np
import pytest

import oracle
from gpu_util import assert_moe_close, bf16_host, dev, guarded_empty, native
from workloads import make_config_inputs, make_moe_inputs

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
    assert m.device_status(clear=True) == 0, "a bounded device wait ran out"


class Fused:
    """Device copies of one workload, tile-layout weight scales, output and workspace."""

    def __init__(self, mx, inp):
        import torch
        self.inp = inp
        self.x = dev(inp.x).view(torch.bfloat16)
        self.ids = dev(inp.topk_ids) if inp.topk_ids is not None else None
        self.w = dev(inp.topk_w) if inp.topk_w is not None else None
        self.w13, self.w2 = dev(inp.w13), dev(inp.w2)
        self.s13t = torch.empty(mx.mxfp4_tiled_scales_bytes(inp.E * 2 * inp.I, inp.H), dtype=torch.uint8,
                                device="cuda")
        self.s2t = torch.empty(mx.mxfp4_tiled_scales_bytes(inp.E * inp.H, inp.I), dtype=torch.uint8, device="cuda")
        mx.mxfp4_scales_to_tiled(dev(inp.s13).view(-1, inp.H // 32), self.s13t)
        mx.mxfp4_scales_to_tiled(dev(inp.s2).view(-1, inp.I // 32), self.s2t)
        self.out = guarded_empty((inp.T, inp.H), torch.bfloat16)
        n = mx.moe_mxfp4_workspace_size(inp.T, inp.H, inp.I, inp.E, inp.K, self.ids is not None)
        self.ws = guarded_empty(max(n, 512), torch.uint8)

    def launch(self, mx, fused, stream=None):
        mx.moe_mxfp4_forward(self.x, self.ids, self.w, self.w13, self.s13t, self.w2, self.s2t, self.out, self.ws,
                             stream=stream, scales_tiled=True, fused=fused)

    def run(self, mx, fused, stream=None):
        self.out.fill_(float("nan"))
        self.launch(mx, fused, stream)
        assert mx.check_workspace(self.ws, stream=stream) == 0, "a bounded device wait ran out"
        return bf16_host(self.out)


def _same_as_multi_kernel(mx, inp, what):
    f = Fused(mx, inp)
    multi = f.run(mx, fused=False)
    one = f.run(mx, fused=True)
    np.testing.assert_array_equal(one, multi, err_msg=what)
    return f, one


def test_tiny_config_bit_identical_and_matches_the_oracle(mx):
    inp = make_config_inputs("tiny")
    _, got = _same_as_multi_kernel(mx, inp, "tiny")
    ref = oracle.moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.w2, inp.s2, inp.I)
    assert_moe_close(got, ref, "fused tiny vs oracle")


def test_routing_edge_cases(mx):
    inp = make_moe_inputs(T=300, H=384, I=256, E=6, K=4, seed=7, routing="uniform", sf_lo=118, sf_hi=126)
    ids = inp.topk_ids
    ids[:, 0] = 2                     # expert 2 gets >= 300 rows: three M tiles
    ids[::7, 1] = -1                  # dropped pairs
    ids[::11, 2] = 6                  # out of range -> dropped
    ids[5] = [-1, -1, -1, -1]         # a token with no valid expert -> zero output
    ids[ids == 4] = 3                 # expert 4 receives nothing
    ids[9] = [1, 1, 3, 3]             # repeated experts in one token
    _, got = _same_as_multi_kernel(mx, inp, "routing edge cases")
    assert ((got[5] & 0x7FFF) == 0).all()


@pytest.mark.parametrize("routing", ["uniform", None])
def test_ragged_k_and_n_tails(mx, routing):
    if routing:
        inp = make_moe_inputs(T=700, H=640, I=384, E=6, K=4, seed=11, routing="uniform")
        inp.topk_ids[::9, 3] = -1
    else:
        inp = make_moe_inputs(T=600, H=640, I=384, E=1, K=1, seed=12, routing=None)
    _same_as_multi_kernel(mx, inp, f"ragged tails, routing={routing}")


@pytest.mark.parametrize("name", ["shared", "decode", "prefill"])
def test_full_size_configs(mx, name):
    _same_as_multi_kernel(mx, make_config_inputs(name), name)


def test_two_calls_in_a_row_and_graph_replay(mx):
    """The barrier counter is re-armed by every call: two calls in a row on one workspace,
    then the call captured in a CUDA graph and replayed twice, all bit-identical."""
    import torch
    inp = make_moe_inputs(T=200, H=512, I=256, E=5, K=3, seed=72, routing="uniform")
    f, first = _same_as_multi_kernel(mx, inp, "first call")
    np.testing.assert_array_equal(f.run(mx, fused=True), first)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        f.launch(mx, True, stream=s)                       # warm up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            f.launch(mx, True, stream=s)
    for _ in range(2):
        f.out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bf16_host(f.out), first)
    assert mx.check_workspace(f.ws) == 0


def test_grid_barrier_wait_runs_out_reports_and_the_context_survives(mx):
    import torch
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mx.selftest_grid_barrier_timeout(ws)
    st = mx.check_workspace(ws)
    dt = time.perf_counter() - t0
    assert st == MX_ERR_DEVICE_TIMEOUT, mx.status_string(st)
    assert 1.0 < dt < 60.0, f"the wait took {dt:.2f} s"
    assert mx.device_status(clear=True) == MX_ERR_DEVICE_TIMEOUT
    assert mx.device_status(clear=True) == 0
    inp = make_config_inputs("tiny")                        # the context still runs the forward
    _same_as_multi_kernel(mx, inp, "after the barrier timeout")
