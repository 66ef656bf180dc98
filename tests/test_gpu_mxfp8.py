"""GPU parity of the MXFP8-activation path against the oracle, through the C ABI (reading
R18: the FP8 reading of the "re-quant" in "Current Bug: vLLM produces empty/garbage output",
"Phase 1: CuTeDSL Shared Expert Kernel"; E4M3 activations with E8M0 scales per 32 over the
MXFP4 weights of "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization").

- act_quant_mxfp8: bit-exact, on random shapes and on special blocks.
- mxfp8_mxfp4_gemm_bf16 (kind::mxf8f6f4): the E4M3 element order and the E2M1 nibble order
  as the tensor core reads them through the spread 4-bit TMA type (one-hot K), the scale
  path (constant codes), and random shapes with ragged M and N against the exact product
  within one BF16 rounding plus the float32 accumulation allowance.
- moe_mxfp4w_mxfp8a_forward: step by step as the MXFP4 forward (tests/moe_check.py): xq/xs
  bit-exact, every re-quantised block admissible, y on the GPU's own decisions, out within
  the per-element bound 2e-2 * max|ref| + 1e-3; tiny, shared, routing edge cases, decode, prefill sample, graph replay.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_gemm_close, assert_moe_close, bf16_host, dev, guarded_empty, native
from moe_check import _ws_view, check_moe_run, tile_edge_tokens
from workloads import f32_to_bf16_bits, make_config_inputs, make_moe_inputs

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

def _quant8(mx, xb):
    import torch
    M, K = xb.shape
    codes = guarded_empty((M, K), torch.uint8)
    sf = guarded_empty((M, K // 32), torch.uint8)
    mx.act_quant_mxfp8(dev(xb).view(torch.bfloat16), codes, sf)
    return codes.cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 32), (37, 288), (300, 7168), (64, 3072)])
def test_act_quant_mxfp8_bit_exact(mx, M, K):
    rng = np.random.default_rng(M * 5 + K)
    x = (rng.standard_normal((M, K)) * np.exp2(rng.uniform(-30, 30, size=(M, 1)))).astype(np.float32)
    xb = f32_to_bf16_bits(x)
    codes, sf = _quant8(mx, xb)
    rq, rs = oracle.act_quant_mxfp8(xb)
    np.testing.assert_array_equal(sf, rs)
    np.testing.assert_array_equal(codes, rq)


def test_act_quant_mxfp8_special_blocks(mx):
    """Zero and -0 blocks, NaN / Inf blocks, the top of the E4M3 range (448, and values that
    saturate), E4M3 ties after scaling, BF16 subnormals and the largest BF16 values."""
    rng = np.random.default_rng(81)
    x = (rng.standard_normal((10, 64)) * 3.0).astype(np.float32)
    x[0] = 0.0
    x[2, 3] = np.nan
    x[3, 40] = -np.inf
    x[4, :32] = np.float32(448.0) * np.array([1, 0.999, 0.5, 0.0625, 1.0 / 1024, -1, 0.75, 0.3] * 4)
    x[5, :32] = np.array([1.0, 1.0625, 1.1875, 3.0 + 1.0 / 16, 2.0 ** -9, 3 * 2.0 ** -10, 0.5, -1.0625] * 4)
    x[6, :32] = np.float32(1e-39)
    x[7, :32] = np.float32(3e38) * np.linspace(-1, 1, 32)
    xb = f32_to_bf16_bits(x)
    xb[1, :32] = 0x8000
    codes, sf = _quant8(mx, xb)
    rq, rs = oracle.act_quant_mxfp8(xb)
    np.testing.assert_array_equal(sf, rs)
    np.testing.assert_array_equal(codes, rq)


# ----------------------------------------------------------------------------- GEMM

def _tiled(mx, sb):
    import torch
    rows, kb = sb.shape
    out = torch.empty(mx.mxfp4_tiled_scales_bytes(rows, 32 * kb), dtype=torch.uint8, device="cuda")
    mx.mxfp4_scales_to_tiled(dev(sb), out)
    return out


def _gemm8(mx, a, sa, b, sb):
    import torch
    M, N = a.shape[0], b.shape[0]
    d = guarded_empty((M, N), torch.bfloat16)
    mx.mxfp8_mxfp4_gemm_bf16(dev(a), dev(sa), dev(b), _tiled(mx, sb), d)
    return bf16_host(d)


def _e4m3_byte(v):
    import torch
    return int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def test_gemm8_one_hot_k(mx):
    """Row m of A is 1.0 at column m mod K and 0 elsewhere, so D[m, n] = B[n, m mod K]: every
    E4M3 element position of A and every E2M1 nibble position of B (lower nibble first, as the
    spread 4-bit TMA type lays them out) must reach the product it belongs to. Bit-exact."""
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(82)
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M) % K] = _e4m3_byte(1.0)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    got = _gemm8(mx, a, sa, b, sb)
    np.testing.assert_array_equal(got, oracle.mxfp8_mxfp4_gemm_bf16(a, sa, b, sb))


def test_gemm8_scale_path_constant_codes(mx):
    """All codes 1.0; every scale byte random: the result is the sum over K blocks of
    32 * 2^(sa + sb - 254), which checks that each MMA reads the scale byte of its own
    32-element block (the scale ids 0..3 of a word) on both sides."""
    M, N, K = 130, 272, 512
    rng = np.random.default_rng(83)
    a = np.full((M, K), _e4m3_byte(1.0), np.uint8)
    b = np.full((N, K // 2), 0x22, np.uint8)                  # E2M1 1.0 in both nibbles
    sa = rng.integers(120, 134, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(120, 134, size=(N, K // 32), dtype=np.uint8)
    got = _gemm8(mx, a, sa, b, sb)
    exact = oracle.mxfp8_values(a, sa) @ oracle.mxfp4_values(b, sb).T
    assert_gemm_close(got, exact, np.abs(exact), "MXFP8 x MXFP4 scale path")


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (77, 272, 512), (300, 512, 1024), (1000, 1024, 7168),
                                   (200, 528, 384)])
def test_gemm8_random(mx, M, N, K):
    rng = np.random.default_rng(M + N + K)
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    a = rng.choice(finite, size=(M, K)).astype(np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(112, 125, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(N, K // 32), dtype=np.uint8)
    got = _gemm8(mx, a, sa, b, sb)
    av, bv = oracle.mxfp8_values(a, sa), oracle.mxfp4_values(b, sb)
    assert_gemm_close(got, av @ bv.T, np.abs(av) @ np.abs(bv).T, f"MXFP8 x MXFP4 {M}x{N}x{K}")


# ----------------------------------------------------------------------------- forward

class Dev8:
    """Device copies of one MoE workload for the MXFP8-activation forward."""

    def __init__(self, mx, inp):
        import torch
        self.inp = inp
        self.x = dev(inp.x).view(torch.bfloat16)
        self.ids = dev(inp.topk_ids) if inp.topk_ids is not None else None
        self.w = dev(inp.topk_w) if inp.topk_w is not None else None
        self.w13, self.w2 = dev(inp.w13), dev(inp.w2)
        self.s13t = _tiled(mx, inp.s13.reshape(-1, inp.H // 32))
        self.s2t = _tiled(mx, inp.s2.reshape(-1, inp.I // 32))
        self.out = guarded_empty((inp.T, inp.H), torch.bfloat16)
        n = mx.moe_mxfp4w_mxfp8a_workspace_size(inp.T, inp.H, inp.I, inp.E, inp.K, self.ids is not None)
        self.ws = guarded_empty(max(n, 512), torch.uint8)

    def launch(self, mx, stream=None):
        mx.moe_mxfp4w_mxfp8a_forward(self.x, self.ids, self.w, self.w13, self.s13t, self.w2, self.s2t, self.out,
                                     self.ws, stream=stream)

    def run(self, mx, stream=None):
        self.launch(mx, stream)
        assert mx.check_workspace(self.ws, stream=stream) == 0, "a bounded device wait ran out"
        return bf16_host(self.out)


def test_mxfp8_tiny_config_full(mx):
    d = Dev8(mx, make_config_inputs("tiny"))
    d.run(mx)
    print("mxfp8 tiny", check_moe_run(mx, d, mxfp8=True))


@pytest.mark.parametrize("T", [1, 37, 200])
def test_mxfp8_shared_small(mx, T):
    d = Dev8(mx, make_moe_inputs(T=T, H=256, I=256, E=1, K=1, seed=100 + T, routing=None))
    d.run(mx)
    print(f"mxfp8 shared T={T}", check_moe_run(mx, d, mxfp8=True))


def test_mxfp8_routing_edges(mx):
    inp = make_moe_inputs(T=300, H=384, I=256, E=6, K=4, seed=7, routing="uniform", sf_lo=118, sf_hi=126)
    ids = inp.topk_ids
    ids[:, 0] = 2
    ids[::7, 1] = -1
    ids[::11, 2] = 6
    ids[5] = [-1, -1, -1, -1]
    ids[ids == 4] = 3
    ids[9] = [1, 1, 3, 3]
    d = Dev8(mx, inp)
    got = d.run(mx)
    print("mxfp8 routing edges", check_moe_run(mx, d, mxfp8=True))
    assert ((got[5] & 0x7FFF) == 0).all()


def test_mxfp8_shared_config_full(mx):
    d = Dev8(mx, make_config_inputs("shared"))
    d.run(mx)
    print("mxfp8 shared T=256", check_moe_run(mx, d, mxfp8=True))


def test_mxfp8_decode_config_full(mx):
    d = Dev8(mx, make_config_inputs("decode"))
    d.run(mx)
    print("mxfp8 decode", check_moe_run(mx, d, mxfp8=True))


def test_mxfp8_prefill_config_sampled(mx):
    inp = make_config_inputs("prefill")
    d = Dev8(mx, inp)
    got = d.run(mx)
    assert np.isfinite((got.astype(np.uint32) << 16).view(np.float32)).all()
    tokens = tile_edge_tokens(inp.topk_ids, inp.E)
    print("mxfp8 prefill", check_moe_run(mx, d, tokens=tokens, mxfp8=True))


def test_mxfp8_graph_replay_bit_identical(mx):
    import torch
    d = Dev8(mx, make_moe_inputs(T=200, H=512, I=256, E=5, K=3, seed=72, routing="uniform"))
    eager = d.run(mx)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d.launch(mx, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        d.out.zero_()
        with torch.cuda.graph(g, stream=s):
            d.launch(mx, stream=s)
    d.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_host(d.out), eager)


def test_mxfp8_nan_tokens_requantise_h_as_positive_nan(mx):
    """Reading R20 in the MXFP8 re-quant: a token whose x holds a NaN (one of each sign) has
    NaN g and u, and its h re-quantises as the positive NaN: scale 255, every E4M3 code 0x7F,
    in a full 32-row warp and in a ragged tile's last warp. Its output row is NaN; every
    other token is within the per-element bound."""
    inp = make_moe_inputs(T=200, H=256, I=256, E=1, K=1, seed=133, routing=None)
    bad = [5, 195]
    inp.x[5, 10] = 0xFFC0
    inp.x[195, 40] = 0x7FC0
    d = Dev8(mx, inp)
    got = d.run(mx)
    T, H, I = inp.T, inp.H, inp.I
    L = mx.moe_mxfp4w_mxfp8a_workspace_layout(T, H, I, 1, 1, False)
    hq = _ws_view(d.ws, L["hq"], T, I)
    hs = _ws_view(d.ws, L["hs"], T, I // 32)
    assert (hq[bad] == 0x7F).all() and (hs[bad] == 255).all()
    g = np.full((1, I), np.nan)
    ref_q, ref_s = oracle.act_quant_mxfp8(oracle.swiglu_bf16(g, g))
    assert (ref_q == 0x7F).all() and (ref_s == 255).all()
    assert np.isnan((got[bad].astype(np.uint32) << 16).view(np.float32)).all()
    good = np.setdiff1d(np.arange(T), bad)
    ref = oracle.moe_mxfp8_forward(inp.x, None, None, inp.w13, inp.s13, inp.w2, inp.s2, inp.I, tokens=good)
    assert_moe_close(got[good], ref, "MXFP8 tokens beside the NaN ones")

