"""Pins for the oracle's activation quantiser and MXFP4 GEMM (CPU only).

The quantiser's rule is the OCP MX v1.0 one (shared exponent floor(log2 amax) - 2, E2M1
round-to-nearest-even saturating at +-6); the pages say only "re-quant" ("Current Bug:
vLLM produces empty/garbage output", "Phase 1: CuTeDSL Shared Expert Kernel"). Its
execution is pinned here by an independent rounding table, a nearest-value search,
math.frexp for the exponent, round trips and invariants. The GEMM is pinned by exact
rational brute force and by a second (integer block) formulation.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import (act_quant_mxfp4, bf16_bits_from_f64, bf16_bits_to_f64, mxfp4_gemm_blockint,
                    mxfp4_gemm_bf16, mxfp4_values, unpack_nibbles)
from workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _cases():
    out = []
    for line in open(os.path.join(GOLDEN, "e2m1_rounding_cases.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            v, c = line.split()
            out.append((float(v), int(c)))
    return out


def _quant_single(v_scaled):
    """Quantise a block whose scale byte is forced to 127 (amax in [4, 8))."""
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 4.0                       # fixes floor(log2 amax) = 2 -> scale byte 127
    x[0, 1] = v_scaled
    codes, sf = act_quant_mxfp4(f32_to_bf16_bits(x))
    assert sf[0, 0] == 127
    return int(unpack_nibbles(codes)[0, 1])


def test_rounding_table():
    for v, code in _cases():
        xb = f32_to_bf16_bits(np.array([v], np.float32))
        if bf16_bits_to_f64(xb)[0] != v:
            continue                     # not a BF16 value; covered by the float path below
        if v >= 8.0:
            continue                     # would change the block scale
        assert _quant_single(v) == code, (v, code)
        assert _quant_single(-v) == (code | 8), (-v, code)


def test_rounding_table_exact_values():
    from oracle.mxfp4_oracle import _e2m1_round_magnitude
    for v, code in _cases():
        assert int(_e2m1_round_magnitude(np.array(v))) == code, (v, code)


def _random_bf16(rng, shape, sigma=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(sigma))


def test_scale_rule_and_nearest_property():
    rng = np.random.default_rng(11)
    xb = _random_bf16(rng, (64, 256), 3.0)
    xb[0, :32] = 0                                            # all-zero block
    xb[1, :32] = 0x8000                                       # all -0 block
    xb[2, :32] = f32_to_bf16_bits(np.full(32, 1e-39, np.float32))   # subnormal amax
    xb[3, 32:64] = f32_to_bf16_bits(np.full(32, 3e38, np.float32))  # huge amax
    codes, sf = act_quant_mxfp4(xb)
    x = bf16_bits_to_f64(xb).reshape(64, 8, 32)
    nib = unpack_nibbles(codes).reshape(64, 8, 32)
    for r in range(64):
        for b in range(8):
            blk = x[r, b]
            amax = float(np.abs(blk).max())
            if amax == 0:
                want = 0
            else:
                m, e = math.frexp(amax)                        # amax = m 2^e, m in [0.5, 1)
                want = min(max((e - 1) - 2 + 127, 0), 254)
            assert sf[r, b] == want, (r, b, amax, sf[r, b], want)
            scale = Fraction(2) ** (int(sf[r, b]) - 127)
            for j in range(32):
                v = Fraction(float(blk[j])) / scale
                c = int(nib[r, b, j])
                assert (c >> 3) == (1 if math.copysign(1.0, blk[j]) < 0 else 0)
                mag = abs(v)
                got = Fraction(GRID[c & 7])
                best = min(abs(Fraction(g) - min(mag, Fraction(6))) for g in GRID)
                assert abs(got - min(mag, Fraction(6))) == best, (r, b, j, float(v), c)
    assert sf[0, 0] == 0 and (nib[0, 0] == 0).all()
    assert sf[1, 0] == 0 and (nib[1, 0] == 8).all()


def test_amax_element_lands_in_4_to_8():
    rng = np.random.default_rng(5)
    xb = _random_bf16(rng, (32, 512), 0.7)
    codes, sf = act_quant_mxfp4(xb)
    x = bf16_bits_to_f64(xb).reshape(32, 16, 32)
    amax = np.abs(x).max(-1)
    scaled = amax / np.ldexp(1.0, sf.astype(np.int64) - 127)
    assert ((scaled >= 4) & (scaled < 8)).all()


def test_round_trip_of_representable_blocks():
    rng = np.random.default_rng(3)
    M, K = 16, 256
    nib = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    nib[:, ::32] = rng.choice([6, 7, 14, 15], size=(M, K // 32))   # every block reaches |4| or |6|
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    sf = rng.integers(100, 150, size=(M, K // 32), dtype=np.uint8)
    vals = mxfp4_values(packed, sf)
    xb = bf16_bits_from_f64(vals)
    codes2, sf2 = act_quant_mxfp4(xb)
    np.testing.assert_array_equal(sf2, sf)
    np.testing.assert_array_equal(mxfp4_values(codes2, sf2), vals)


def test_nonfinite_block():
    xb = np.zeros((1, 64), np.uint16)
    xb[0, 3] = 0x7FC0                   # NaN in block 0
    xb[0, 40] = 0xFF80                  # -inf in block 1
    xb[0, 41] = 0x3F80                  # 1.0 (positive) in block 1
    codes, sf = act_quant_mxfp4(xb)
    nib = unpack_nibbles(codes)[0]
    assert sf.tolist() == [[255, 255]]
    assert nib[40] == 15 and nib[41] == 7 and nib[0] == 7


def _brute_gemm(a_codes, a_sf, b_codes, b_sf):
    """Exact rational A.B^T from the bit definitions, no numpy arithmetic."""
    def val(codes, sf, r, c):
        byte = int(codes[r, c // 2])
        n = (byte & 15) if c % 2 == 0 else (byte >> 4)
        s, e, m = n >> 3, (n >> 1) & 3, n & 1
        mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
        return (-mag if s else mag) * Fraction(2) ** (int(sf[r, c // 32]) - 127)
    M, K = a_codes.shape[0], 2 * a_codes.shape[1]
    N = b_codes.shape[0]
    A = [[val(a_codes, a_sf, i, k) for k in range(K)] for i in range(M)]
    B = [[val(b_codes, b_sf, j, k) for k in range(K)] for j in range(N)]
    return [[sum(A[i][k] * B[j][k] for k in range(K)) for j in range(N)] for i in range(M)]


def test_gemm_brute_force_tiny():
    rng = np.random.default_rng(9)
    M, N, K = 3, 5, 96
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(118, 127, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 127, size=(N, K // 32), dtype=np.uint8)
    exact = _brute_gemm(a, sa, b, sb)
    got = mxfp4_gemm_bf16(a, sa, b, sb)
    fp = mxfp4_values(a, sa) @ mxfp4_values(b, sb).T
    for i in range(M):
        for j in range(N):
            assert Fraction(fp[i, j]) == exact[i][j]               # float64 path is exact
            assert got[i, j] == bf16_bits_from_f64(np.array([float(exact[i][j])]))[0]
    # transposition: (A.B^T)^T = B.A^T
    np.testing.assert_array_equal(mxfp4_gemm_bf16(b, sb, a, sa), got.T)


def test_gemm_two_formulations_agree():
    rng = np.random.default_rng(10)
    M, N, K = 24, 40, 512
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(110, 140, size=(M, K // 32), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(N, K // 32), dtype=np.uint8)
    fp = mxfp4_values(a, sa) @ mxfp4_values(b, sb).T
    bi = mxfp4_gemm_blockint(a, sa, b, sb)
    np.testing.assert_array_equal(fp, bi)
