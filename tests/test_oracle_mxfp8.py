"""Pins of the oracle's MXFP8 activation functions (reading R18: the OCP MX rule with E4M3
elements, the FP8 variant of the pages' "re-quant", "Current Bug: vLLM produces
empty/garbage output", "Phase 1: CuTeDSL Shared Expert Kernel").

Each check compares the oracle with something other than itself: torch's float32 ->
float8_e4m3fn conversion, round trips of representable blocks, a brute-force quantiser in
exact rationals whose E4M3 grid is built from the bit fields, and the MoE invariants.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from workloads import f32_to_bf16_bits, make_moe_inputs


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def test_elements_match_torch_e4m3_of_the_scaled_block():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(81)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.uniform(-20, 20, size=(64, 1)))).astype(np.float32)
    xb = _bits(x)
    q, sf = oracle.act_quant_mxfp8(xb)
    xv = oracle.bf16_bits_to_f64(xb).reshape(64, 8, 32)
    v = np.clip(xv * np.ldexp(1.0, 127 - sf.astype(np.int64))[..., None], -448, 448).astype(np.float32)
    ref = torch.from_numpy(v.reshape(64, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)


def test_scale_puts_the_block_maximum_in_the_top_binade():
    """Unclamped, amax * 2^(127 - E) lies in [256, 512): E4M3's largest binade, so the rule
    subtracts 8 (E4M3's largest exponent), not E2M1's 2."""
    rng = np.random.default_rng(82)
    x = (rng.standard_normal((32, 512)) * np.exp2(rng.uniform(-30, 30, size=(32, 1)))).astype(np.float32)
    xb = _bits(x)
    _, sf = oracle.act_quant_mxfp8(xb)
    amax = np.abs(oracle.bf16_bits_to_f64(xb)).reshape(32, 16, 32).max(-1)
    t = amax * np.ldexp(1.0, 127 - sf.astype(np.int64))
    assert ((t >= 256) & (t < 512)).all()


def test_round_trip_of_representable_blocks():
    rng = np.random.default_rng(83)
    M, K = 16, 256
    code = rng.integers(0, 127, size=(M, K)).astype(np.uint8) | (rng.integers(0, 2, size=(M, K)) << 7).astype(np.uint8)
    code[:, ::32] = (0x78 + rng.integers(0, 7, size=(M, K // 32))).astype(np.uint8)   # 256 .. 448 per block
    E = rng.integers(100, 140, size=(M, K // 32)).astype(np.uint8)
    x = oracle.e4m3fn_decode(code) * np.repeat(np.ldexp(1.0, E.astype(np.int64) - 127), 32, axis=1)
    xb = _bits(x)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(xb), x)          # exact in BF16
    q, sf = oracle.act_quant_mxfp8(xb)
    np.testing.assert_array_equal(sf, E)
    np.testing.assert_array_equal(q, code)


def test_special_blocks():
    x = np.zeros((5, 32), np.float32)
    x[2, 3] = np.nan
    x[3, 7] = -np.inf
    x[4, :] = 1e-39                                     # subnormal: the scale clamps at 0
    xb = _bits(x)
    xb[1] = 0x8000
    q, sf = oracle.act_quant_mxfp8(xb)
    assert sf[0, 0] == 0 and (q[0] == 0).all()
    assert sf[1, 0] == 0 and (q[1] == 0x80).all()
    assert sf[2, 0] == 255 and q[2, 3] in (0x7F, 0xFF) and q[2, 0] == 0x7F
    assert sf[3, 0] == 255 and q[3, 7] == 0xFF
    assert sf[4, 0] == 0
    v = oracle.bf16_bits_to_f64(xb[4]) * 2.0 ** 127                     # about 0.17
    np.testing.assert_array_equal(oracle.e4m3fn_decode(q[4]), oracle.e4m3fn_decode(oracle.e4m3_round_code(v)))


# ----------------------------------------------------------------------------- brute force

def _e4m3_grid():
    """Non-negative finite E4M3 values from the bit fields, as exact rationals."""
    out = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            out.append(Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return out


_GRID = _e4m3_grid()


def _quant_block8(vals):
    """Brute-force MXFP8 quantisation of 32 exact values: their dequantised values."""
    amax = max(abs(v) for v in vals)
    if amax == 0:
        return [Fraction(0)] * 32
    e = math.floor(math.log2(amax))
    while Fraction(2) ** e > amax:
        e -= 1
    while Fraction(2) ** (e + 1) <= amax:
        e += 1
    E = min(max(e - 8 + 127, 0), 254)
    scale = Fraction(2) ** (E - 127)
    out = []
    for v in vals:
        m = min(abs(v) / scale, Fraction(448))
        d = [abs(m - g) for g in _GRID]
        best = min(d)
        idx = [i for i in range(len(_GRID)) if d[i] == best]
        i = idx[0] if len(idx) == 1 else [j for j in idx if j % 2 == 0][0]
        out.append(_GRID[i] * scale * (-1 if v < 0 else 1))
    return out


def _mx4_row(codes_row, sf_row):
    out = []
    for c in range(2 * len(codes_row)):
        b = int(codes_row[c // 2])
        n = (b & 15) if c % 2 == 0 else (b >> 4)
        s, e, m = n >> 3, (n >> 1) & 3, n & 1
        mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
        out.append((-mag if s else mag) * Fraction(2) ** (int(sf_row[c // 32]) - 127))
    return out


def _bf16(q):
    if q == 0:
        return Fraction(0)
    a = abs(q)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 7)
    n = a / quantum
    fl = math.floor(n)
    rem = n - fl
    r = fl + 1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2) else fl
    return r * quantum * (1 if q > 0 else -1)


@pytest.mark.parametrize("routed", [True, False])
def test_moe_mxfp8_brute_force_tiny(routed):
    if routed:
        inp = make_moe_inputs(T=3, H=64, I=32, E=3, K=2, seed=84, routing="uniform", sf_lo=120, sf_hi=126)
    else:
        inp = make_moe_inputs(T=2, H=64, I=32, E=1, K=1, seed=85, routing=None, sf_lo=120, sf_hi=126)
    got = oracle.bf16_bits_to_f64(oracle.moe_mxfp8_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13,
                                                           inp.w2, inp.s2, inp.I))
    I, H = inp.I, inp.H
    for t in range(inp.T):
        xs = [Fraction(float(v)) for v in oracle.bf16_bits_to_f64(inp.x[t])]
        xq = sum((_quant_block8(xs[b:b + 32]) for b in range(0, H, 32)), [])
        acc = [Fraction(0)] * H
        for k in range(inp.K):
            e = int(inp.topk_ids[t, k]) if routed else 0
            wgt = Fraction(float(inp.topk_w[t, k])) if routed else Fraction(1)
            W13 = [_mx4_row(inp.w13[e, r], inp.s13[e, r]) for r in range(2 * I)]
            gu = [sum(a * b for a, b in zip(xq, W13[r])) for r in range(2 * I)]
            g = [_bf16(v) for v in gu[:I]]
            u = [_bf16(v) for v in gu[I:]]
            h = [_bf16(Fraction(float(a) / (1.0 + math.exp(-float(a)))) * b) for a, b in zip(g, u)]
            hq = sum((_quant_block8(h[b:b + 32]) for b in range(0, I, 32)), [])
            W2 = [_mx4_row(inp.w2[e, r], inp.s2[e, r]) for r in range(H)]
            y = [_bf16(sum(a * b for a, b in zip(hq, W2[r]))) for r in range(H)]
            acc = [a + wgt * yy for a, yy in zip(acc, y)]
        np.testing.assert_array_equal(got[t], np.array([float(_bf16(a)) for a in acc]))


def test_moe_mxfp8_shared_equals_single_expert_routing():
    inp = make_moe_inputs(T=4, H=64, I=32, E=1, K=1, seed=86, routing=None)
    shared = oracle.moe_mxfp8_forward(inp.x, None, None, inp.w13, inp.s13, inp.w2, inp.s2, inp.I)
    routed = oracle.moe_mxfp8_forward(inp.x, np.zeros((4, 1), np.int32), np.ones((4, 1), np.float32), inp.w13,
                                      inp.s13, inp.w2, inp.s2, inp.I)
    np.testing.assert_array_equal(shared, routed)


def test_mxfp8_is_closer_to_bf16_than_mxfp4():
    """The accuracy side of the trade-off: on the same inputs the MXFP8-activation forward is
    nearer the unquantised-activation result than the MXFP4 one (cosine)."""
    inp = make_moe_inputs(T=8, H=256, I=128, E=4, K=2, seed=87, routing="uniform")
    ref = oracle.bf16_bits_to_f64(oracle.moe_mxfp8_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13,
                                                           inp.w2, inp.s2, inp.I))
    four = oracle.bf16_bits_to_f64(oracle.moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13,
                                                      inp.w2, inp.s2, inp.I))
    # unquantised activations: the exact products of x and of h with the MXFP4 weights
    xv = oracle.bf16_bits_to_f64(inp.x)
    exact = np.zeros_like(ref)
    for t in range(inp.T):
        for k in range(inp.K):
            e = inp.topk_ids[t, k]
            gu = xv[t] @ oracle.mxfp4_values(inp.w13[e], inp.s13[e]).T
            g, u = gu[:inp.I], gu[inp.I:]
            h = g / (1 + np.exp(-g)) * u
            exact[t] += float(inp.topk_w[t, k]) * (h @ oracle.mxfp4_values(inp.w2[e], inp.s2[e]).T)

    def cos(a, b):
        return float(a.ravel() @ b.ravel() / (np.linalg.norm(a) * np.linalg.norm(b)))
    assert cos(ref, exact) > cos(four, exact)


def test_mxfp8_mxfp4_gemm_brute_force():
    """The mixed GEMM against exact rationals from the bit fields of both formats."""
    rng = np.random.default_rng(88)
    M, N, K = 3, 4, 64
    a = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x10                                     # no NaN codes
    sa = rng.integers(115, 135, size=(M, K // 32), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(N, K // 32), dtype=np.uint8)
    grid = _e4m3_grid()
    got = oracle.bf16_bits_to_f64(oracle.mxfp8_mxfp4_gemm_bf16(a, sa, b, sb))
    for i in range(M):
        av = [(-1 if a[i, k] >> 7 else 1) * grid[int(a[i, k]) & 0x7F] * Fraction(2) ** (int(sa[i, k // 32]) - 127)
              for k in range(K)]
        for j in range(N):
            bv = _mx4_row(b[j], sb[j])
            assert got[i, j] == float(_bf16(sum(x * y for x, y in zip(av, bv)))), (i, j)
