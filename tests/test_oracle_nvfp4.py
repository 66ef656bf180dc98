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


# ----------------------------------------------------------------------------- quantiser (R15)

def _f32_bits(v):
    return np.asarray(v, np.float32).view(np.uint32)


def test_e4m3_round_code_matches_torch():
    """The oracle's E4M3 encoder (a search of its own value table) against torch's float32 ->
    float8_e4m3fn conversion, on every E4M3 value, every midpoint (ties), the float32
    neighbours of each midpoint, and log-uniform samples down to the subnormals."""
    torch = pytest.importorskip("torch")
    vals = oracle.e4m3fn_decode(np.arange(127)).astype(np.float32)
    mids = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)   # exact in float32
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    rng = np.random.default_rng(41)
    samp = np.exp2(rng.uniform(-12, np.log2(448.0), 20000)).astype(np.float32)
    a = np.concatenate([vals, mids, near, samp, np.float32([0, 2.0 ** -10, 2.0 ** -11, 447.9, 448])])
    a = a[(a >= 0) & (a <= 448)]
    ref = torch.from_numpy(a).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_round_code(a.astype(np.float64)), ref)


def _bf16_bits_of(v):
    torch = pytest.importorskip("torch")
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_round_trip_of_representable_blocks():
    """x = LUT[c] * e4m3(S) * g with a +-6 code in every block and g a power of two: the
    quantiser must give back exactly (c, S) -- its scale is amax / (6 g), its codes x / (S g),
    lower nibble first, sign kept (including -0)."""
    rng = np.random.default_rng(43)
    M, K = 24, 128
    lut = oracle.e2m1_decode(np.arange(16))
    for g in (1.0, 2.0 ** -9, 2.0 ** 7):
        code = rng.integers(0, 16, size=(M, K)).astype(np.uint8)
        code[:, ::16] = rng.choice([7, 15], size=(M, K // 16))          # a +-6 per block
        S = rng.integers(0x08, 0x77, size=(M, K // 16)).astype(np.uint8)  # normal E4M3
        x = lut[code] * np.repeat(oracle.e4m3fn_decode(S), 16, axis=1) * g
        xb = _bf16_bits_of(x)
        np.testing.assert_array_equal(oracle.bf16_bits_to_f64(xb), x)     # exact in BF16
        q, sf = oracle.nvfp4_quantize(xb, g)
        np.testing.assert_array_equal(sf, S)
        np.testing.assert_array_equal(q, (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8))


def test_quantize_scale_is_nearest_e4m3_of_amax_over_6g():
    """In float64: the decoded scale is the E4M3 value nearest amax / (6 g) (within the float32
    rounding of the two products), clamped at 448; so 6 * scale * g covers the block's amax
    to E4M3 precision."""
    rng = np.random.default_rng(44)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.uniform(-6, 6, size=(64, 1)))).astype(np.float32)
    xb = _bf16_bits_of(x)
    g = float(np.float32(3.7e-3))
    _, sf = oracle.nvfp4_quantize(xb, g)
    amax = np.abs(oracle.bf16_bits_to_f64(xb)).reshape(64, 16, 16).max(-1)
    t = np.minimum(amax / (6.0 * g), 448.0)
    grid = oracle.e4m3fn_decode(np.arange(127))
    dist = np.abs(grid[None, None, :] - t[..., None])
    got = np.abs(oracle.e4m3fn_decode(sf) - t)
    assert (got <= dist.min(-1) + t * 2.0 ** -22).all()


def test_quantize_codes_nearest_scaled_value():
    """Each code is the E2M1 value nearest x / (scale * g) (ties excepted, where the float32
    steps decide), saturating at 6."""
    rng = np.random.default_rng(45)
    x = (rng.standard_normal((32, 512)) * 3.0).astype(np.float32)
    xb = _bf16_bits_of(x)
    g = float(np.float32(0.0131))
    q, sf = oracle.nvfp4_quantize(xb, g)
    xv = oracle.bf16_bits_to_f64(xb)
    v = np.abs(xv) / (np.repeat(oracle.e4m3fn_decode(sf), 16, axis=1) * g)
    nib = oracle.unpack_nibbles(q)
    mags = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    d_all = np.abs(np.minimum(v, 6.0)[..., None] - mags)
    d_got = np.abs(np.minimum(v, 6.0) - mags[nib & 7])
    tie = np.sort(d_all, -1)[..., 1] - np.sort(d_all, -1)[..., 0] < 1e-6
    assert ((d_got <= d_all.min(-1) + 1e-12) | tie).all()
    assert ((nib >> 3) == np.signbit(xv)).all()


def test_quantize_special_blocks():
    g = 0.01
    rows = np.zeros((6, 16), np.float32)
    rows[1, :] = -0.0
    rows[2, :8] = 1e-8                                            # amax / (6 g) below 2^-10: scale 0
    rows[3, 3] = np.nan
    rows[4, 5] = -np.inf
    rows[5, :] = np.linspace(-1e4, 1e4, 16)                       # amax / (6 g) above 448: clamped
    xb = _bf16_bits_of(rows)
    xb[1] = 0x8000
    q, sf = oracle.nvfp4_quantize(xb, g)
    nib = oracle.unpack_nibbles(q)
    assert sf[0, 0] == 0 and (nib[0] == 0).all()
    assert sf[1, 0] == 0 and (nib[1] == 8).all()
    assert sf[2, 0] == 0 and (nib[2] == 0).all()
    assert sf[3, 0] == 0x7F and sf[4, 0] == 0x7F
    assert (nib[3] == ((np.signbit(oracle.bf16_bits_to_f64(xb[3])) << 3) | 7)).all()
    assert nib[4, 5] == 15 and nib[4, 0] == 7
    assert sf[5, 0] == 0x7E and nib[5, 0] == 15 and nib[5, 15] == 7   # 448, codes saturate at 6


# ----------------------------------------------------------------------------- NVFP4 MoE (R16)

def _bf16_exact(q):
    """Nearest BF16 (ties to even) of a finite exact rational, in the normal range."""
    import math
    from fractions import Fraction
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


def _nv_row(codes_row, sf_row):
    return [_nv_exact(codes_row[None], sf_row[None], 0, c) for c in range(2 * len(codes_row))]


@pytest.mark.parametrize("routed", [True, False])
def test_moe_nvfp4_brute_force_tiny(routed):
    """Exact rationals for every GEMM, global and weighted sum; the quantiser and SiLU
    (pinned above and in the MXFP4 tests) are taken from the oracle."""
    import math
    from fractions import Fraction
    from workloads import make_nvfp4_moe_inputs
    if routed:
        inp = make_nvfp4_moe_inputs(T=3, H=64, I=32, E=3, K=2, seed=51, routing="uniform")
    else:
        inp = make_nvfp4_moe_inputs(T=2, H=64, I=32, E=1, K=1, seed=52, routing=None)
    got = oracle.bf16_bits_to_f64(oracle.moe_nvfp4_forward(
        inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.g13, inp.w2, inp.s2, inp.g2,
        inp.x_global, inp.h_global, inp.I))
    F = lambda v: Fraction(float(np.float32(v)))                     # noqa: E731
    I, H = inp.I, inp.H
    for t in range(inp.T):
        xq, xs = oracle.nvfp4_quantize(inp.x[t:t + 1], inp.x_global)
        xv = _nv_row(xq[0], xs[0])
        acc = [Fraction(0)] * H
        for k in range(inp.K):
            e = int(inp.topk_ids[t, k]) if routed else 0
            wgt = F(inp.topk_w[t, k]) if routed else Fraction(1)
            W13 = [_nv_row(inp.w13[e, r], inp.s13[e, r]) for r in range(2 * I)]
            gu = [sum(a * b for a, b in zip(xv, W13[r])) for r in range(2 * I)]
            g = [_bf16_exact(v * F(inp.x_global) * F(inp.g13[e, 0])) for v in gu[:I]]
            u = [_bf16_exact(v * F(inp.x_global) * F(inp.g13[e, 1])) for v in gu[I:]]
            h = [_bf16_exact(Fraction(float(a) / (1.0 + math.exp(-float(a)))) * b) for a, b in zip(g, u)]
            hb = np.array([oracle.bf16_bits_from_f64(np.array([float(v)]))[0] for v in h], np.uint16)
            hq, hs = oracle.nvfp4_quantize(hb[None], inp.h_global)
            hv = _nv_row(hq[0], hs[0])
            W2 = [_nv_row(inp.w2[e, r], inp.s2[e, r]) for r in range(H)]
            y = [_bf16_exact(sum(a * b for a, b in zip(hv, W2[r])) * F(inp.h_global) * F(inp.g2[e]))
                 for r in range(H)]
            acc = [a + wgt * yy for a, yy in zip(acc, y)]
        want = np.array([float(_bf16_exact(a)) for a in acc])
        np.testing.assert_array_equal(got[t], want)


def _nv_forward(inp, **over):
    a = dict(x=inp.x, ids=inp.topk_ids, w=inp.topk_w, g13=inp.g13, g2=inp.g2, gx=inp.x_global, gh=inp.h_global)
    a.update(over)
    return oracle.moe_nvfp4_forward(a["x"], a["ids"], a["w"], inp.w13, inp.s13, a["g13"], inp.w2, inp.s2,
                                    a["g2"], a["gx"], a["gh"], inp.I)


def test_moe_nvfp4_global_placement():
    """Where each global enters. (1) Doubling x's global halves every scale byte's value and
    leaves x's dequantised values, so the output, unchanged: the global is applied in L1.
    (2) Doubling the up globals doubles h exactly; with h's global doubled too its codes and
    scales are unchanged, and halving w2's globals restores y. (3) Doubling only the gate
    globals changes the output (SiLU is not linear), so gate and up are not interchangeable."""
    from workloads import make_nvfp4_moe_inputs
    inp = make_nvfp4_moe_inputs(T=6, H=128, I=64, E=3, K=2, seed=53, routing="uniform")
    base = _nv_forward(inp)
    np.testing.assert_array_equal(_nv_forward(inp, gx=2 * inp.x_global), base)
    g13 = inp.g13.copy()
    g13[:, 1] *= 2
    np.testing.assert_array_equal(_nv_forward(inp, g13=g13, gh=2 * inp.h_global, g2=inp.g2 / 2), base)
    g13 = inp.g13.copy()
    g13[:, 0] *= 2
    assert (_nv_forward(inp, g13=g13) != base).any()
    assert (_nv_forward(inp, g2=inp.g2 * 2) != base).any()


def test_moe_nvfp4_shared_equals_single_expert_routing():
    from workloads import make_nvfp4_moe_inputs
    inp = make_nvfp4_moe_inputs(T=5, H=64, I=32, E=1, K=1, seed=54, routing=None)
    shared = _nv_forward(inp)
    routed = _nv_forward(inp, ids=np.zeros((5, 1), np.int32), w=np.ones((5, 1), np.float32))
    np.testing.assert_array_equal(shared, routed)


# ----------------------------------------------------------------------------- fused projection (R17)

def test_gemm_segments_brute_force_exact_rationals():
    """Two stacked weight matrices with their own globals (q_a and kv of the pages' fused
    projection): every output is the exact rational sum times a_global * b_global[segment],
    rounded once; a segment boundary inside a 16-column block is allowed."""
    from fractions import Fraction
    rng = np.random.default_rng(27)
    M, K = 3, 32
    seg = [5, 3, 8]
    N = sum(seg)
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa = rng.integers(0x20, 0x50, size=(M, K // 16), dtype=np.uint8)
    sb = rng.integers(0x20, 0x50, size=(N, K // 16), dtype=np.uint8)
    ga, gbs = np.float32(0.0371), [np.float32(1.5e-3), np.float32(-2.0 ** -9), np.float32(7.25)]
    got = oracle.bf16_bits_to_f64(oracle.nvfp4_gemm_segments_bf16(a, sa, ga, b, sb, gbs, seg))
    bounds = np.cumsum([0] + seg)
    for i in range(M):
        for j in range(N):
            s_idx = int(np.searchsorted(bounds, j, side="right")) - 1
            exact = sum(_nv_exact(a, sa, i, k) * _nv_exact(b, sb, j, k) for k in range(K))
            exact *= Fraction(float(ga)) * Fraction(float(gbs[s_idx]))
            want = oracle.bf16_bits_to_f64(oracle.bf16_bits_from_f64(np.array([float(exact)])))[0]
            assert got[i, j] == want, (i, j)


def test_gemm_segments_single_segment_is_the_gemm():
    rng = np.random.default_rng(28)
    a = rng.integers(0, 256, size=(4, 64), dtype=np.uint8)
    b = rng.integers(0, 256, size=(32, 64), dtype=np.uint8)
    sa = rng.integers(0x20, 0x50, size=(4, 8), dtype=np.uint8)
    sb = rng.integers(0x20, 0x50, size=(32, 8), dtype=np.uint8)
    np.testing.assert_array_equal(oracle.nvfp4_gemm_segments_bf16(a, sa, 0.5, b, sb, [0.25], [32]),
                                  oracle.nvfp4_gemm_bf16(a, sa, 0.5, b, sb, 0.25))


# ----------------------------------------------------------------------------- calibration (R19)

def _e4m3_byte(v):
    import torch
    return int(torch.tensor([v], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def test_calibrated_global_maps_the_largest_input_to_the_largest_nvfp4_value():
    """With the calibrated global, the block holding the batch's largest |x| gets the largest
    E4M3 scale (448, torch's encoding) and that element the largest E2M1 code (6.0, the OCP
    table), the dequantised value equals that |x| up to the float32 rounding of the global,
    and no block's scale goes past 448: the whole range is used, nothing is clipped."""
    rng = np.random.default_rng(191)
    from workloads import f32_to_bf16_bits
    x = (rng.standard_normal((37, 256)) * np.exp2(rng.uniform(-6, 6, size=(37, 1)))).astype(np.float32)
    xb = f32_to_bf16_bits(x)
    g = oracle.nvfp4_activation_global([xb])
    q, sf = oracle.nvfp4_quantize(xb, g)
    xv = oracle.bf16_bits_to_f64(xb)
    r, c = np.unravel_index(np.argmax(np.abs(xv)), xv.shape)
    top = _e4m3_byte(448.0)
    assert sf[r, c // 16] == top
    assert (sf <= top).all()
    nib = oracle.unpack_nibbles(q)[r, c]
    table = _e2m1_table()
    assert abs(table[nib & 7]) == 6.0
    deq = 6.0 * 448.0 * g
    assert abs(deq - abs(xv[r, c])) <= abs(xv[r, c]) * 2.0 ** -23


def test_calibration_running_maximum_skips_non_finite_and_clamps():
    from workloads import f32_to_bf16_bits
    rng = np.random.default_rng(192)
    xb = f32_to_bf16_bits(rng.standard_normal((60, 64)).astype(np.float32) * 3)
    whole = oracle.nvfp4_activation_global([xb])
    parts = [xb[:10], xb[10:45], xb[45:]]
    assert oracle.nvfp4_activation_global(parts) == whole
    assert oracle.nvfp4_activation_global(parts[::-1]) == whole
    bad = xb.copy()
    bad[3, 5], bad[7, 9], bad[8, 1] = 0x7FC0, 0x7F80, 0xFF80           # NaN, +inf, -inf
    assert oracle.nvfp4_activation_global([bad]) == whole
    assert oracle.nvfp4_activation_global([np.zeros((4, 16), np.uint16)]) == 2.0 ** -117
    big = f32_to_bf16_bits(np.full((1, 16), 1e35, np.float32))
    assert oracle.nvfp4_activation_global([big]) == float(np.float32(2.0 ** 100))
    # one float32 division, nearest even: the largest finite BF16 magnitude of 1.5 gives
    # 1.5 / 2688 rounded once
    one = f32_to_bf16_bits(np.array([[1.5, -0.25] + [0.0] * 14], np.float32))
    assert oracle.nvfp4_activation_global([one]) == float(np.float32(1.5) / np.float32(2688.0))


def test_generator_global_is_the_calibration_of_its_batch():
    from workloads import make_nvfp4_config_inputs
    inp = make_nvfp4_config_inputs("tiny")
    assert inp.x_global == oracle.nvfp4_activation_global([inp.x])
