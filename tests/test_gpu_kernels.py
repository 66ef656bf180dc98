"""GPU parity of the single kernels against the CPU oracle, through the C ABI.

Bit-exact: MXFP4 -> BF16 dequant, NVFP4 -> BF16 dequant, FP8 128x128 dequant, the MX
activation quantiser (codes and scales) and the routing permutation. The block-scaled GEMM is compared with the exact
product (one BF16 rounding plus the float32 accumulation allowance), first on structured
inputs that isolate the data path (all scales 1) and the scale-factor path (all codes
equal), then on random inputs across tile, stage and ragged-edge boundaries.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_gemm_close, bf16_host, dev, guarded_empty, native
from workloads import f32_to_bf16_bits, make_dequant_inputs, make_nvfp4_scales

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


def _empty(shape, dtype):
    """An output buffer with canary guard bands, checked after the test."""
    return guarded_empty(shape, dtype)


# ----------------------------------------------------------------------------- dequant

@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 64), (257, 96), (1000, 7168)])
def test_mxfp4_dequant_bit_exact(mx, rows, cols):
    import torch
    rng = np.random.default_rng(rows * 7 + cols)
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    sf = rng.integers(0, 256, size=(rows, cols // 32), dtype=np.uint8)   # every scale byte incl. 0, 255
    out = _empty((rows, cols), torch.bfloat16)
    mx.mxfp4_dequant(dev(codes), dev(sf), out)
    np.testing.assert_array_equal(bf16_host(out), oracle.mxfp4_dequant(codes, sf))


def test_mxfp4_dequant_all_code_scale_pairs(mx):
    import torch
    codes = np.tile(np.arange(256, dtype=np.uint8).reshape(16, 16), (256, 1))  # 4096 rows x 32 cols
    sf = np.repeat(np.arange(256, dtype=np.uint8), 16).reshape(4096, 1)
    out = _empty((4096, 32), torch.bfloat16)
    mx.mxfp4_dequant(dev(codes), dev(sf), out)
    np.testing.assert_array_equal(bf16_host(out), oracle.mxfp4_dequant(codes, sf))


@pytest.mark.parametrize("g", [1.0, 0.000372, -3.5, 2.0 ** -140, 1.0e37, float("inf")])
def test_nvfp4_dequant_all_code_scale_pairs(mx, g):
    """Every (code, E4M3 scale byte) pair, including the NaN bytes, at globals that give
    float32 subnormals (2^-140), overflow (1e37), a negative sign and an infinity."""
    import torch
    nib = np.arange(16, dtype=np.uint8)
    codes = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), (256, 1))   # 256 rows x 16 cols
    sf = np.arange(256, dtype=np.uint8).reshape(256, 1)
    out = _empty((256, 16), torch.bfloat16)
    mx.nvfp4_dequant(dev(codes), dev(sf), g, out)
    np.testing.assert_array_equal(bf16_host(out), oracle.nvfp4_dequant(codes, sf, g))


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 48), (257, 1040), (2048, 7168)])
def test_nvfp4_dequant_bit_exact(mx, rows, cols):
    import torch
    rng = np.random.default_rng(rows * 11 + cols)
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    sf = rng.integers(0, 256, size=(rows, cols // 16), dtype=np.uint8)   # every E4M3 byte incl. NaN
    out = _empty((rows, cols), torch.bfloat16)
    mx.nvfp4_dequant(dev(codes), dev(sf), 0.0123, out)
    np.testing.assert_array_equal(bf16_host(out), oracle.nvfp4_dequant(codes, sf, 0.0123))


def test_nvfp4_dequant_full_size_sampled(mx):
    """The 48 experts' w13 codes with NVFP4 scales, as the bench times them; sampled rows."""
    import torch
    w13, _, _, _, _, _ = make_dequant_inputs()
    n13, _, g = make_nvfp4_scales()
    R, half = w13.shape
    out = _empty((R, 2 * half), torch.bfloat16)
    mx.nvfp4_dequant(dev(w13), dev(n13), g, out)
    rows = np.unique(np.concatenate([np.random.default_rng(98).integers(0, R, 48), [0, R - 1]]))
    got = bf16_host(out[torch.from_numpy(rows).cuda()])
    np.testing.assert_array_equal(got, oracle.nvfp4_dequant(w13[rows], n13[rows], g))


# units of 16 columns per row: 1, 17, 65, a power of two (32) and 3 over many block rows
@pytest.mark.parametrize("rows,cols", [(1, 16), (130, 272), (300, 1040), (257, 512), (2049, 48)])
def test_fp8_dequant_bit_exact(mx, rows, cols):
    import torch
    rng = np.random.default_rng(rows + cols)
    q = rng.integers(0, 256, size=(rows, cols), dtype=np.uint8)          # includes NaN codes
    sf = rng.integers(0, 256, size=((rows + 127) // 128, (cols + 127) // 128), dtype=np.uint8)
    out = _empty((rows, cols), torch.bfloat16)
    mx.fp8_block_dequant_128x128(dev(q), dev(sf), out)
    np.testing.assert_array_equal(bf16_host(out), oracle.fp8_block_dequant_128x128(q, sf))


def test_dequant_sweep_full_size_sampled(mx):
    """The full dequant workload (48 experts, FP8 [7168, 7168]); sampled rows vs the oracle."""
    import torch
    w13, s13, w2, s2, q, fsf = make_dequant_inputs()
    rng = np.random.default_rng(99)
    for codes, sf in ((w13, s13), (w2, s2)):
        R, half = codes.shape
        out = _empty((R, 2 * half), torch.bfloat16)
        mx.mxfp4_dequant(dev(codes), dev(sf), out)
        rows = np.unique(np.concatenate([rng.integers(0, R, 48), [0, R - 1]]))
        got = bf16_host(out[torch.from_numpy(rows).cuda()])
        np.testing.assert_array_equal(got, oracle.mxfp4_dequant(codes[rows], sf[rows]))
        del out
    out = _empty(q.shape, torch.bfloat16)
    mx.fp8_block_dequant_128x128(dev(q), dev(fsf), out)
    rows = np.unique(np.concatenate([rng.integers(0, q.shape[0], 64), [0, q.shape[0] - 1]]))
    ref = oracle.fp8_block_dequant_128x128(q, fsf)[rows]
    np.testing.assert_array_equal(bf16_host(out)[rows], ref)


# ----------------------------------------------------------------------------- act quant

@pytest.mark.parametrize("M,K", [(1, 32), (5, 96), (300, 7168), (2048, 3072)])
def test_act_quant_bit_exact(mx, M, K):
    import torch
    rng = np.random.default_rng(M * 3 + K)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(2.0)
    x[rng.random((M, K)) < 0.01] *= 1000.0
    xb = f32_to_bf16_bits(x)
    specials = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x7F7F, 0xFF7F, 0x3E80, 0x3F40,
                         0x3FA0, 0x3FE0, 0x4020, 0x4060, 0x40A0], dtype=np.uint16)
    flat = xb.reshape(-1)
    flat[: min(flat.size, 4096)][rng.random(min(flat.size, 4096)) < 0.2] = rng.choice(specials)
    if M >= 5:
        xb[1, :32] = 0                     # all-zero block
        xb[2, :32] = 0x8000                # all -0 block
        xb[3, 3] = 0x7FC0                  # NaN block
        xb[4, 40] = 0xFF80                 # -inf block
    codes = _empty((M, K // 2), torch.uint8)
    sf = _empty((M, K // 32), torch.uint8)
    mx.act_quant_mxfp4(dev(xb).view(torch.bfloat16), codes, sf)
    ref_c, ref_s = oracle.act_quant_mxfp4(xb)
    np.testing.assert_array_equal(sf.cpu().numpy(), ref_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)


# ----------------------------------------------------------------------------- GEMM

def _tiled(mx, sb):
    import torch
    rows, kb = sb.shape
    out = _empty(mx.mxfp4_tiled_scales_bytes(rows, 32 * kb), torch.uint8)
    mx.mxfp4_scales_to_tiled(dev(sb), out)
    return out


def _tiled_layout_reference(sf):
    """The tile layout written out with numpy indexing (block (g, w): byte l*16 + j*4 + b is
    the scale of row 128g + 32j + l, K block 4w + b; rows past the end are 0)."""
    rows, kb = sf.shape
    G, KW = (rows + 127) // 128, kb // 4
    padded = np.zeros((G * 128, kb), np.uint8)
    padded[:rows] = sf
    t = padded.reshape(G, 4, 32, KW, 4)          # g, j, l, w, b
    return t.transpose(0, 3, 2, 1, 4).reshape(-1)  # g, w, l, j, b


@pytest.mark.parametrize("rows,cols", [(1, 128), (128, 7168), (300, 3072), (6144, 1024)])
def test_scales_to_tiled_bit_exact(mx, rows, cols):
    rng = np.random.default_rng(rows + cols)
    sf = rng.integers(0, 256, size=(rows, cols // 32), dtype=np.uint8)
    got = _tiled(mx, sf).cpu().numpy()
    np.testing.assert_array_equal(got, _tiled_layout_reference(sf))


def _gemm_case(mx, a, sa, b, sb, what):
    import torch
    M, N = a.shape[0], b.shape[0]
    d = _empty((M, N), torch.bfloat16)
    mx.mxfp4_gemm_bf16(dev(a), dev(sa), dev(b), _tiled(mx, sb), d)
    A = oracle.mxfp4_values(a, sa)
    B = oracle.mxfp4_values(b, sb)
    exact = A @ B.T
    absdot = np.abs(A) @ np.abs(B).T
    assert_gemm_close(bf16_host(d), exact, absdot, what)


def test_gemm_data_path_unit_scales(mx):
    """All scales 1: isolates operand layout, swizzle, nibble order and K advance."""
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 256
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    _gemm_case(mx, a, sa, b, sb, "unit scales")


def test_gemm_one_hot_k(mx):
    """A single nonzero K column: checks which element of the byte the tensor core reads
    first (lower nibble = even column) and the K position of every MMA of a stage."""
    M, N, K = 128, 256, 256
    for k in (0, 1, 63, 64, 127, 130, 255):
        a = np.zeros((M, K // 2), np.uint8)
        b = np.zeros((N, K // 2), np.uint8)
        code = 0x02 if k % 2 == 0 else 0x20              # value 1.0 in column k
        a[:, k // 2] = code
        b[:, k // 2] = code
        b[::3, k // 2] = 0x04 if k % 2 == 0 else 0x40    # 2.0 on every third B row
        sa = np.full((M, K // 32), 127, np.uint8)
        sb = np.full((N, K // 32), 127, np.uint8)
        _gemm_case(mx, a, sa, b, sb, f"one-hot k={k}")


def test_gemm_scale_path_constant_codes(mx):
    """All codes 1.0: D[m, n] = 32 * sum_kb 2^(sa[m,kb] + sb[n,kb] - 254) isolates the
    scale-factor layout (rows, K blocks, sf ids)."""
    rng = np.random.default_rng(2)
    M, N, K = 128, 256, 512
    a = np.full((M, K // 2), 0x22, np.uint8)
    b = np.full((N, K // 2), 0x22, np.uint8)
    sa = rng.integers(117, 138, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(117, 138, size=(N, K // 32), dtype=np.uint8)
    _gemm_case(mx, a, sa, b, sb, "constant codes")


# A GEMM with fewer than 152 work units of 128 x 256 runs 128-column tiles; the last two
# shapes (160 units) run 256-column tiles.
@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (128, 256, 128), (77, 256, 1024), (300, 512, 2048),
                                   (129, 272, 384), (1000, 1024, 7168), (513, 7168, 3072),
                                   (1280, 4096, 512), (2048, 2560, 384)])
def test_gemm_random(mx, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(115, 135, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(N, K // 32), dtype=np.uint8)
    _gemm_case(mx, a, sa, b, sb, f"random {M}x{N}x{K}")


def _nv_tiled(mx, sf):
    import torch
    rows, kb = sf.shape
    out = _empty(mx.nvfp4_tiled_scales_bytes(rows, 16 * kb), torch.uint8)
    mx.nvfp4_scales_to_tiled(dev(sf), out)
    return out


def test_nvfp4_scales_to_tiled_bit_exact(mx):
    rng = np.random.default_rng(31)
    sf = rng.integers(0, 256, size=(300, 7168 // 16), dtype=np.uint8)
    np.testing.assert_array_equal(_nv_tiled(mx, sf).cpu().numpy(), _tiled_layout_reference(sf))


# NVFP4 scales are read as unsigned E4M3 by the tensor core: the inputs keep the sign bit clear.
@pytest.mark.parametrize("M,N,K,ga,gb", [(128, 256, 256, 1.0, 1.0), (77, 272, 512, 0.0123, 2.5),
                                         (300, 512, 1024, 3.0e-3, -0.7), (1000, 1024, 7168, 0.05, 0.02),
                                         (200, 512, 384, 0.01, 0.5), (64, 256, 128, 1.0, 1.0)])
def test_nvfp4_gemm_random(mx, M, N, K, ga, gb):
    import torch
    rng = np.random.default_rng(M + N + K)
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x50, size=(M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x28, 0x48, size=(N, K // 16), dtype=np.uint8)
    d = _empty((M, N), torch.bfloat16)
    mx.nvfp4_gemm_bf16(dev(a), dev(sa), ga, dev(b), _nv_tiled(mx, sb), gb, d)
    exact = oracle.nvfp4_gemm_f64(a, sa, ga, b, sb, gb)
    absdot = np.abs(oracle.nvfp4_values(a, sa, 1.0)) @ np.abs(oracle.nvfp4_values(b, sb, 1.0)).T
    absdot *= abs(float(np.float32(ga)) * float(np.float32(gb)))
    assert_gemm_close(bf16_host(d), exact, absdot, f"nvfp4 {M}x{N}x{K}")


def test_nvfp4_gemm_scale_words_one_hot(mx):
    """All codes 1.0 and all scales 1.0 except one E4M3 scale per row of A: D[m, n] picks
    out which 16-column block (which scale word and which of its four bytes) each MMA
    reads, for every one of the stage's four words."""
    import torch
    M, N, K = 128, 256, 512
    a = np.full((M, K // 2), 0x22, np.uint8)
    b = np.full((N, K // 2), 0x22, np.uint8)
    sa = np.full((M, K // 16), 0x38, np.uint8)
    sb = np.full((N, K // 16), 0x38, np.uint8)
    sa[np.arange(M), np.arange(M) % (K // 16)] = 0x40                   # scale 2.0 at block m mod 32
    sb[np.arange(N), (3 * np.arange(N)) % (K // 16)] = 0x30             # scale 0.5 at block 3n mod 32
    d = _empty((M, N), torch.bfloat16)
    mx.nvfp4_gemm_bf16(dev(a), dev(sa), 1.0, dev(b), _nv_tiled(mx, sb), 1.0, d)
    np.testing.assert_array_equal(bf16_host(d), oracle.nvfp4_gemm_bf16(a, sa, 1.0, b, sb, 1.0))


# ----------------------------------------------------------------------------- routing

# one chunk of at most 2048 pairs (routed in one CTA: 1, 400, exactly 2048 and 2046 pairs, the
# last with the largest E) and several chunks
@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (100, 4, 5), (256, 8, 48), (341, 6, 1024), (3000, 8, 48),
                                   (8192, 8, 48), (513, 6, 300)])
def test_route_bit_exact(mx, T, K, E):
    import torch
    rng = np.random.default_rng(T + K + E)
    ids = rng.integers(-1, E + 1, size=(T, K)).astype(np.int32)      # includes dropped ids
    if T >= 100:
        ids[: T // 2, 0] = 0                                          # one expert with many tiles
    ws = _empty(mx.moe_mxfp4_workspace_size(T, 128, 128, E, K, True), torch.uint8)
    counts = _empty((E,), torch.int32)
    offsets = _empty((E + 1,), torch.int32)
    row_of = _empty((T, K), torch.int32)
    mx.moe_mxfp4_route(dev(ids), E, counts, offsets, row_of, ws)
    rc, ro, rr, _ = oracle.moe_route(ids, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(row_of.cpu().numpy(), rr)


@pytest.mark.parametrize("M,K,seg", [(300, 7168, [1536, 576]), (130, 512, [48, 208, 16, 272]),
                                     (64, 384, [256]), (200, 256, [16] * 8)])
def test_nvfp4_fused_projection(mx, M, K, seg):
    """Weights stacked along N with one global per segment (the fused q_a + kv projection):
    segment boundaries inside 256-column tiles and inside 32-column pieces, up to eight
    segments, against the oracle within the GEMM bound."""
    import torch
    rng = np.random.default_rng(M + K + len(seg))
    N = sum(seg)
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x50, size=(M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x28, 0x48, size=(N, K // 16), dtype=np.uint8)
    ga = 0.0173
    gbs = [float(np.float32(v)) for v in rng.uniform(1e-4, 4.0, size=len(seg)) * rng.choice([-1, 1], len(seg))]
    d = _empty((M, N), torch.bfloat16)
    mx.nvfp4_gemm_bf16_multi(dev(a), dev(sa), ga, dev(b), _nv_tiled(mx, sb), gbs, seg, d)
    g = np.repeat([float(np.float32(ga)) * v for v in gbs], seg)
    S = oracle.nvfp4_values(a, sa, 1.0) @ oracle.nvfp4_values(b, sb, 1.0).T
    absdot = np.abs(oracle.nvfp4_values(a, sa, 1.0)) @ np.abs(oracle.nvfp4_values(b, sb, 1.0)).T
    got = bf16_host(d)
    assert_gemm_close(got, S * g[None, :], absdot * np.abs(g)[None, :], f"fused projection {seg}")
    ref = oracle.nvfp4_gemm_segments_bf16(a, sa, ga, b, sb, gbs, seg)
    assert (got == ref).mean() > 0.98
