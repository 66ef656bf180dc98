"""Pins of the oracle's NVFP4 functions (readings R11, R12; "Current Bug: vLLM produces
empty/garbage output", "What we know": NVFP4 weights dequantised to BF16; same page,
"Phase 2: CuTeDSL Attention Kernel": per-tensor global scales).

Each check compares the oracle with something other than itself:
- torch's float8_e4m3fn decoding, float32 multiplication and float32 -> bfloat16 rounding,
  applied to every (code, scale byte) pair;
- the MXFP4 oracle, for scale bytes that are powers of two;
- one-hot tensors, for nibble order and for the 16 columns each scale covers.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    """The 16 E2M1 values from the OCP MX table fixture (independent of the oracle)."""
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_table.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            vals[int(parts[0], 0)] = float(parts[-1])
    return np.array([vals[i] for i in range(16)], np.float32)


def _all_pairs():
    """codes [256, 8]: row r holds the 16 nibbles 0..15 (lower nibble first); sf [256, 1] = r."""
    nib = np.arange(16, dtype=np.uint8)
    row = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    return np.tile(row, (256, 1)), np.arange(256, dtype=np.uint8).reshape(256, 1)


@pytest.mark.parametrize("g", [1.0, 0.000372, -3.5, 2.0 ** -140, 1.0e37, 3.0e-41, np.inf])
def test_dequant_matches_float32_library_arithmetic(g):
    torch = pytest.importorskip("torch")
    codes, sf = _all_pairs()
    got = oracle.nvfp4_dequant(codes, sf, g)
    lut = torch.from_numpy(_e2m1_table())                                   # [16]
    scale = torch.from_numpy(sf.reshape(-1)).view(torch.float8_e4m3fn).to(torch.float32)
    prod = lut.reshape(1, 16) * scale.reshape(256, 1)                      # exact in float32
    ref = (prod * torch.tensor(np.float32(g))).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(oracle.bf16_bits_to_f64(got))
    ref_nan = np.isnan(oracle.bf16_bits_to_f64(ref))
    np.testing.assert_array_equal(nan, ref_nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_power_of_two_scales_equal_mxfp4():
    """E4M3 bytes with a zero mantissa and a normal exponent e encode 2^(e-7), which is the
    E8M0 byte 120 + e: with global 1 both formats must give the same BF16 values."""
    rng = np.random.default_rng(11)
    R, C = 64, 256
    codes = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    e = rng.integers(1, 15, size=(R, C // 32))
    e4 = (e << 3).astype(np.uint8)
    sf16 = np.repeat(e4, 2, axis=1)
    e8 = (120 + e).astype(np.uint8)
    np.testing.assert_array_equal(oracle.nvfp4_dequant(codes, sf16, 1.0), oracle.mxfp4_dequant(codes, e8))


def test_scale_covers_its_16_columns_and_lower_nibble_first():
    R, C = 4, 64
    codes = np.full((R, C // 2), 0x22, np.uint8)                 # every value 1.0
    sf = np.full((R, C // 16), 0x38, np.uint8)                   # every scale 1.0
    base = oracle.nvfp4_values(codes, sf, 1.0)
    for b in range(C // 16):
        s2 = sf.copy()
        s2[1, b] = 0x40                                          # 2.0
        diff = oracle.nvfp4_values(codes, s2, 1.0) != base
        cols = np.nonzero(diff[1])[0]
        assert list(cols) == list(range(16 * b, 16 * b + 16)) and not diff[[0, 2, 3]].any()
    c2 = codes.copy()
    c2[0, 0] = 0x02                                              # column 0 -> 1.0, column 1 -> 0
    v = oracle.nvfp4_values(c2, sf, 1.0)
    assert v[0, 0] == 1.0 and v[0, 1] == 0.0


def test_nan_sign_rule():
    # nibbles 8 (-0) and 9 (-0.5); the NaN's sign is the XOR of code, scale and global signs
    codes = np.array([[0x98] * 8], np.uint8)
    for sbyte, g, neg in ((0x7F, 1.0, True), (0xFF, 1.0, False), (0x38, np.nan, True),
                          (0x38, -np.inf, False)):
        got = oracle.nvfp4_dequant(codes, np.array([[sbyte]], np.uint8), g)
        assert got[0, 0] == (0xFFC0 if neg else 0x7FC0), (hex(sbyte), g, hex(int(got[0, 0])))


def _nv_exact(codes, sf, r, c):
    """Exact rational value of NVFP4 element (r, c) with global 1, from the bit fields."""
    from fractions import Fraction
    byte = int(codes[r, c // 2])
    n = (byte >> 4) if c % 2 else (byte & 15)
    s, e, m = n >> 3, (n >> 1) & 3, n & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    sb = int(sf[r, c // 16])
    se, ee, me = sb >> 7, (sb >> 3) & 15, sb & 7
    smag = Fraction(me, 8) * Fraction(2) ** -6 if ee == 0 else (1 + Fraction(me, 8)) * Fraction(2) ** (ee - 7)
    return (-1) ** (s ^ se) * mag * smag


def test_gemm_brute_force_exact_rationals():
    from fractions import Fraction
    rng = np.random.default_rng(21)
    M, N, K = 3, 4, 48
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x08, 0x7E, size=(M, K // 16), dtype=np.uint8)    # finite, positive
    sb = rng.integers(0x88, 0xFE, size=(N, K // 16), dtype=np.uint8)    # finite, negative
    ga, gb = np.float32(0.375), np.float32(-1.5e-3)
    got = oracle.nvfp4_gemm_f64(a, sa, ga, b, sb, gb)
    for i in range(M):
        for j in range(N):
            exact = sum(_nv_exact(a, sa, i, k) * _nv_exact(b, sb, j, k) for k in range(K))
            exact *= Fraction(float(ga)) * Fraction(float(gb))
            assert got[i, j] == float(exact)            # the exact value, rounded once


def test_gemm_power_of_two_scales_equal_mxfp4():
    """With E4M3 scales 2^(e-7) (repeated over both 16-column halves of each 32-block) and
    globals 1, the NVFP4 GEMM is the MXFP4 GEMM with E8M0 bytes 120 + e."""
    rng = np.random.default_rng(23)
    M, N, K = 8, 16, 256
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    ea = rng.integers(1, 15, size=(M, K // 32))
    eb = rng.integers(1, 15, size=(N, K // 32))
    got = oracle.nvfp4_gemm_bf16(a, np.repeat((ea << 3).astype(np.uint8), 2, axis=1), 1.0,
                                 b, np.repeat((eb << 3).astype(np.uint8), 2, axis=1), 1.0)
    ref = oracle.mxfp4_gemm_bf16(a, (120 + ea).astype(np.uint8), b, (120 + eb).astype(np.uint8))
    np.testing.assert_array_equal(got, ref)
