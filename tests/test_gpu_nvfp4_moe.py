"""GPU parity of the NVFP4 activation quantiser and moe_nvfp4_forward against the CPU
oracle, through the C ABI (readings R15, R16: the NVFP4 variant of the expert FFN with the
activation global of "Phase 1: CuTeDSL Shared Expert Kernel" and the separate gate/up
weight globals of "Phase 2: CuTeDSL Attention Kernel", page "Current Bug: vLLM produces
empty/garbage output").

The quantiser is bit-exact. The forward is checked step by step as the MXFP4 one is
(tests/moe_check.py): xq/xs bit-exact, every re-quantised block admissible, y on the GPU's
own decisions, out within |err| <= 2e-2 * max|ref| + 1e-3 with cosine >= 0.9999.
"""
import numpy as np
import pytest

import oracle
from gpu_util import bf16_host, dev, guarded_empty, native
from moe_check import check_nvfp4_moe_run, tile_edge_tokens
from workloads import f32_to_bf16_bits, make_nvfp4_config_inputs, make_nvfp4_moe_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mx():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    m = native()
    assert m.device_status(clear=True) == 0
    yield m
    assert m.device_status(clear=True) == 0, "a bounded device wait ran out"


# ----------------------------------------------------------------------------- quantiser

def _quant_gpu(mx, xb, g):
    import torch
    M, K = xb.shape
    codes = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    mx.act_quant_nvfp4(dev(xb).view(torch.bfloat16), g, codes, sf)
    return codes.cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("M,K,g", [(1, 16, 1.0), (37, 272, 0.0123), (300, 7168, 0.00191), (64, 3072, 0.25),
                                   (5, 1024, 2.0 ** -110), (9, 512, 2.0 ** 90)])
def test_act_quant_nvfp4_bit_exact(mx, M, K, g):
    rng = np.random.default_rng(M * 7 + K)
    x = (rng.standard_normal((M, K)) * np.exp2(rng.uniform(-8, 8, size=(M, 1)))).astype(np.float32)
    xb = f32_to_bf16_bits(x)
    codes, sf = _quant_gpu(mx, xb, g)
    rq, rs = oracle.nvfp4_quantize(xb, g)
    np.testing.assert_array_equal(sf, rs)
    np.testing.assert_array_equal(codes, rq)


def test_act_quant_nvfp4_special_blocks(mx):
    """Zero and -0 blocks, blocks whose scale rounds to 0, NaN / Inf blocks, saturated scales,
    ties of the E2M1 rounding (values at midpoints after scaling), subnormal BF16 inputs."""
    rng = np.random.default_rng(61)
    g = 0.01
    x = (rng.standard_normal((12, 64)) * 2.0).astype(np.float32)
    x[0] = 0.0
    x[2, :16] = 1e-9
    x[3, 5] = np.nan
    x[4, 17] = -np.inf
    x[5, :16] = np.linspace(-1e5, 1e5, 16)
    x[6, :16] = np.float32(6 * 448 * g) * np.array([1, .25, .75, .125, .375, .625, .875, 5 / 6] * 2)
    x[7, :16] = np.float32(1e-39)
    xb = f32_to_bf16_bits(x)
    xb[1] = 0x8000
    codes, sf = _quant_gpu(mx, xb, g)
    rq, rs = oracle.nvfp4_quantize(xb, g)
    np.testing.assert_array_equal(sf, rs)
    np.testing.assert_array_equal(codes, rq)


# ----------------------------------------------------------------------------- forward

class NvDev:
    """Device copies of one NVFP4 MoE workload (weight scales in the tile layout)."""

    def __init__(self, mx, inp):
        import torch
        self.inp = inp
        self.x = dev(inp.x).view(torch.bfloat16)
        self.ids = dev(inp.topk_ids) if inp.topk_ids is not None else None
        self.w = dev(inp.topk_w) if inp.topk_w is not None else None
        self.w13, self.w2, self.g13, self.g2 = (dev(a) for a in (inp.w13, inp.w2, inp.g13, inp.g2))
        self.s13t = torch.empty(mx.nvfp4_tiled_scales_bytes(inp.E * 2 * inp.I, inp.H), dtype=torch.uint8,
                                device="cuda")
        self.s2t = torch.empty(mx.nvfp4_tiled_scales_bytes(inp.E * inp.H, inp.I), dtype=torch.uint8, device="cuda")
        mx.nvfp4_scales_to_tiled(dev(inp.s13.reshape(-1, inp.H // 16)), self.s13t)
        mx.nvfp4_scales_to_tiled(dev(inp.s2.reshape(-1, inp.I // 16)), self.s2t)
        self.out = guarded_empty((inp.T, inp.H), torch.bfloat16)
        n = mx.moe_nvfp4_workspace_size(inp.T, inp.H, inp.I, inp.E, inp.K, self.ids is not None)
        self.ws = guarded_empty(max(n, 256), torch.uint8)

    def launch(self, mx, stream=None):
        inp = self.inp
        mx.moe_nvfp4_forward(self.x, self.ids, self.w, self.w13, self.s13t, self.g13, self.w2, self.s2t, self.g2,
                             inp.x_global, inp.h_global, self.out, self.ws, stream=stream)

    def run(self, mx, stream=None):
        self.launch(mx, stream)
        assert mx.check_workspace(self.ws, stream=stream) == 0, "a bounded device wait ran out"
        return bf16_host(self.out)


def test_nvfp4_tiny_config_full(mx):
    d = NvDev(mx, make_nvfp4_config_inputs("tiny"))
    d.run(mx)
    print("nvfp4 tiny", check_nvfp4_moe_run(mx, d))


@pytest.mark.parametrize("T", [1, 100, 300])
def test_nvfp4_shared_small(mx, T):
    d = NvDev(mx, make_nvfp4_moe_inputs(T=T, H=512, I=256, E=1, K=1, seed=70 + T, routing=None))
    d.run(mx)
    print(f"nvfp4 shared T={T}", check_nvfp4_moe_run(mx, d))


def test_nvfp4_ragged_tails_and_routing_edges(mx):
    """H = 640: L1's last K stage holds 128 (two of four scale words) and L2's last N tile
    128 columns; I = 384: L2's last K stage holds 128. Dropped ids, experts over several
    ragged 128-row tiles, an expert nobody picks."""
    inp = make_nvfp4_moe_inputs(T=500, H=640, I=384, E=7, K=4, seed=71, routing="uniform")
    inp.topk_ids[::7, 2] = -1
    inp.topk_ids[inp.topk_ids == 6] = 5
    inp.topk_ids[3, :] = -1
    d = NvDev(mx, inp)
    first = d.run(mx)
    print("nvfp4 ragged", check_nvfp4_moe_run(mx, d))
    assert (first[3] == 0).all()
    np.testing.assert_array_equal(d.run(mx), first)             # deterministic


def test_nvfp4_shared_config_full(mx):
    d = NvDev(mx, make_nvfp4_config_inputs("shared"))
    d.run(mx)
    print("nvfp4 shared T=256", check_nvfp4_moe_run(mx, d))


def test_nvfp4_decode_config_full(mx):
    d = NvDev(mx, make_nvfp4_config_inputs("decode"))
    d.run(mx)
    print("nvfp4 decode", check_nvfp4_moe_run(mx, d))           # all 64 tokens


def test_nvfp4_prefill_config_sampled(mx):
    """The NVFP4 routed prefill forward the bench reports (T = 8192, 48 experts, top-8, Zipf
    routing), on every expert's first and last M tile and the tiles scheduled last."""
    inp = make_nvfp4_config_inputs("prefill")
    d = NvDev(mx, inp)
    got = d.run(mx)
    assert np.isfinite((got.astype(np.uint32) << 16).view(np.float32)).all()
    tokens = tile_edge_tokens(inp.topk_ids, inp.E)
    assert tokens.size >= 64
    print("nvfp4 prefill", check_nvfp4_moe_run(mx, d, tokens=tokens))


def test_nvfp4_graph_capture_replays_bit_identical(mx):
    import torch
    d = NvDev(mx, make_nvfp4_moe_inputs(T=200, H=512, I=256, E=5, K=3, seed=72, routing="uniform"))
    eager = d.run(mx)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d.run(mx, stream=s)                                   # warm up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        d.out.zero_()
        with torch.cuda.graph(g, stream=s):
            d.launch(mx, stream=s)                            # no host read-back while capturing
    d.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_host(d.out), eager)


# ----------------------------------------------------------------------------- calibration

def test_nvfp4_calibrate_global_bit_exact(mx):
    """The device calibration (running maximum of the finite |x| over warm-up batches, then
    amax / (6 * 448) in float32) equals the oracle's (reading R19), bit for bit: batches of
    odd sizes (a scalar tail after the 16-byte vectors), NaN and infinities skipped, an
    empty batch, and the running maximum carried across calls."""
    import torch
    rng = np.random.default_rng(93)
    shapes = [(3, 37), (64, 7168), (0, 16), (5, 8), (1000, 96)]
    batches = []
    for i, (M, K) in enumerate(shapes):
        x = (rng.standard_normal((M, K)) * np.exp2(rng.uniform(-20, 20, size=(M, 1)))).astype(np.float32)
        xb = f32_to_bf16_bits(x)
        if M > 2:
            xb[1, 2], xb[2, 0] = 0x7FC0, 0xFF80                  # NaN, -inf: skipped
        batches.append(xb)
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    for i, xb in enumerate(batches):
        xd = dev(xb).view(torch.bfloat16) if xb.size else torch.empty(xb.shape, dtype=torch.bfloat16, device="cuda")
        mx.nvfp4_calibrate_global(xd, amax, g)
        want = oracle.nvfp4_activation_global(batches[: i + 1])
        assert float(g.cpu()[0]) == want, (i, float(g.cpu()[0]), want)
    finite = np.concatenate([oracle.bf16_bits_to_f64(b).ravel() for b in batches])
    assert float(amax.cpu()[0]) == np.abs(finite[np.isfinite(finite)]).max()


def test_nvfp4_forward_with_the_device_calibrated_global(mx):
    """The activation global the forward runs with comes from the device calibration of the
    batch itself (no host-side numpy step): it equals the workload's, and the forward checks
    out step by step against the oracle with it."""
    import torch
    inp = make_nvfp4_config_inputs("tiny")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    mx.nvfp4_calibrate_global(dev(inp.x).view(torch.bfloat16), amax, g)
    x_global = float(g.cpu()[0])
    assert x_global == inp.x_global
    inp.x_global = x_global
    d = NvDev(mx, inp)
    d.run(mx)
    print("nvfp4 tiny, device-calibrated global", check_nvfp4_moe_run(mx, d))
