"""Plain CPU oracle (numpy, float64) for the mixture-of-experts expert FFN over FP4 weights
(MXFP4, and the NVFP4 and MXFP8-activation variants).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import or run this module. It shares no code with the
CUDA path: no tables, no helpers, no constants; it imports numpy only.

Sources (page title -- section):

[FMT]  "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization" -- "FP4 (E2M1) expert weight format
       confirmed": w1/w3 int8 [3072, 3584] with E8M0 [3072, 224] -> [3072, 7168]
       (224 * 32 = 7168); w2 int8 [7168, 1536] with E8M0 [7168, 96] -> [7168, 3072]
       (96 * 32 = 3072); nibble index 0 is +0.0 and index 8 is -0.0.
[DQ]   same page -- "Script update: dequant_fp8_to_bf16.py now handles ALL compressed types":
       item 1, FP8 weights dequantised block-wise (128 x 128) as float8_e4m3fn x
       float8_e8m0fnu scale -> BF16; item 2, FP4 (E2M1) expert weights: two values per
       byte, lower nibble first, E2M1 LUT lookup x E8M0 scale, one scale per row per 32
       columns (MXFP4 microscaling), output 2x the stored columns -> BF16.
[PIPE] "Current Bug: vLLM produces empty/garbage output" -- "Phase 1: CuTeDSL Shared Expert
       Kernel": L1 GEMM -> SiLU -> re-quant -> L2 GEMM; the MoE adds routing, top-k and
       scatter; gate_up_proj is stacked as in the MoE L1; the shared expert is the MoE
       with one group and no routing.
[BF16] same page -- "Phase 3: Clean up": BF16 only where it must be (SiLU activation,
       final scatter).
[DG]   "2026-05-11 -- DeepSeek V4 NVFP4 vLLM Serving: Full End-to-End" -- "What We Fixed",
       item 1: FP8 block scales with quant_block_shape=(128, 128) and use_e8m0=True.
[NVQ]  "Current Bug: vLLM produces empty/garbage output" -- "What we know", "Confirmed
       working": all NVFP4 weights dequantise correctly to BF16 (a standalone test).
[GS]   same page -- "Phase 2: CuTeDSL Attention Kernel": a projection carries a per-tensor
       global scale (weight_scale_2); the MoE's gate and up carry different ones.

Element formats follow the OCP Microscaling (MX) v1.0 definitions of E2M1, E8M0 and the
E4M3 ("fn": no infinities, S.1111.111 is NaN) encoding; the pages name the formats but
print no bit layout.

Readings where the pages are silent:

R1  The first activation quantisation uses the same MXFP4 rule as the re-quant: "re-quant"
    in [PIPE] presupposes an earlier quantisation of x, and both GEMM operands are E2M1.
R2  The re-quant rule is the OCP MX one: shared exponent floor(log2(amax)) - 2 (2 is the
    largest E2M1 exponent), biased by 127 and clamped to [0, 254]; elements rounded to
    E2M1 to nearest, ties to even, saturating at +-6; the sign is kept (so -0 -> code 8).
    A block holding a NaN or an infinity gets scale byte 255 and codes sign|7.
R3  The L1 outputs g (gate) and u (up) are rounded to BF16 before SiLU, and h =
    SiLU(g) * u is rounded to BF16 before the re-quant ([BF16]). The L2 output y is
    rounded to BF16 before the weighted scatter. The oracle computes every product and
    sum exactly (float64; the dot products of MXFP4 values are exact), rounds once per
    stated BF16 step, and evaluates SiLU in float64.
R4  In the stacked w13, rows [0, I) are the gate (w1) and rows [I, 2I) the up (w3).
R5  The weighted scatter sums w[t, k] * y[t, k] over the slots k = 0..K-1 in float64 and
    rounds once to BF16. An expert id outside [0, E) (e.g. -1, "not on this rank")
    contributes nothing. With no routing (shared expert) out = y.
R6  FP8 block dequant multiplies by the block scale ([DQ] item 1 says weight x block_scale).
R7  A NaN result is written as the quiet NaN 0x7FC0 with the element's sign bit (E2M1
    code bit 3, E4M3 bit 7); infinities and overflow follow BF16 round-to-nearest-even.
R8  The BF16 rounding of an exact value is round-to-nearest, ties to even, with BF16
    subnormals (BF16 has float32's exponent range).
R11 An NVFP4 tensor ([NVQ], [GS]; the pages print no layout) holds E2M1 codes packed as in
    MXFP4 (two per byte, lower nibble first), one E4M3 ("fn") scale per 16 columns and one
    float32 global scale per tensor; its value is LUT[code] * e4m3(scale) * global.
R12 NVFP4 -> BF16 rounds the exact product once to float32 and then to BF16, both to
    nearest-even: what float32 arithmetic gives, since LUT[code] * e4m3(scale) is exact in
    float32. A NaN result (a NaN scale byte, a NaN global, or 0 times an infinite global)
    is 0x7FC0 with the XOR of the code's, the scale's and the global's sign bits.
R14 The NVFP4 GEMM is the exact sum of the scaled E2M1 products times the product of the
    two float32 globals, rounded once to BF16 (the pages give one global per operand and
    do not say where it is applied). R13, the GEMM's unsigned scale bytes, is a limit of
    the GPU path's inputs; the oracle decodes every byte.
R15 NVFP4 quantisation of a row with float32 global scale g ("Warmup-based gs
    computation" in [GS]'s plan: g is fixed before the call, not taken from the data),
    per 16-column block, every step a float32 operation rounded to nearest even:
    r = 1 / (6 g); amax = max |x|; S = the E4M3 byte nearest to min(amax * r, 448), ties
    to the even code; d = e4m3(S) * g; each element's code is E2M1(x * (1 / d)) to nearest,
    ties to even, saturating at +-6, sign kept. S = 0 gives codes sign|0. A block holding
    a NaN or an infinity gets S = 0x7F (NaN) and codes sign|7. This is the published NVFP4
    encoder (scale = amax / 6 per block, relative to the global); the float32 order is a
    reading, chosen so that both sides take every rounding decision in the same precision.
R16 The NVFP4 MoE forward is the MXFP4 one (R1, R3-R5) with NVFP4 in every quantised
    step: x is quantised with the activation global g_x, h with g_h (R15); the gate and up
    halves of an expert's w13 carry their own globals ([GS]: "gate+up with different gs"),
    w2 one; L1's g = bf16(sum * g_x * g_gate) and u = bf16(sum * g_x * g_up), L2's
    y = bf16(sum * g_h * g_w2), each product of two float32 globals exact in float64 and
    applied once to the exact sum (R14).
R17 A fused projection (the pages' q_a + kv weights stacked along N, each with its own
    weight_scale_2, [GS]) is one NVFP4 GEMM over the stacked B whose output columns of
    segment s are scaled by a_global * b_global[s] (R14 per segment).
R18 MXFP8 activations (E4M3 elements, one E8M0 scale per 32; the pages do not name this
    variant, it is the FP8 reading of "re-quant"): the OCP MX rule with E4M3's largest
    exponent 8 in place of E2M1's 2 -- scale byte E = clamp(floor(log2 amax) - 8 + 127,
    0, 254) (0 for amax = 0); element = E4M3 nearest x * 2^(127 - E), ties to even,
    saturating at +-448, sign kept (-0 -> 0x80); a block holding a NaN or an infinity gets
    E = 255 and elements sign|0x7F. The MXFP8 MoE forward is R1, R3-R5 with MXFP8 in both
    activation quantisations and the MXFP4 weights unchanged.
R19 The warm-up-based activation global ([GS]'s "warmup-based gs"; the pages give no
    formula): the largest finite |x| over the calibration batches, divided by 6 * 448 (the
    largest NVFP4 magnitude) in one float32 division, clamped into R15's range. NaN and
    infinities are skipped (a non-finite input would leave no usable global).
R20 A NaN in h (from a NaN g or u, from SiLU(-inf) = -inf / inf, or from 0 * inf) is the
    positive quiet NaN 0x7FC0, so the re-quant codes it sign 0 (E2M1 code 7, E4M3 0x7F).
    Float arithmetic gives a NaN it generates no defined sign, and the pages cover no
    non-finite values; R7's "sign of the element" applies where the inputs define that
    sign (the dequants).

Parity status: every function below is pinned by the ``-m "not gpu"`` tests (tables from
the OCP MX definitions and torch's float8 conversions, one-hot nibble/scale tests, the
shape identities printed on the pages, brute force with exact rationals on tiny inputs,
and invariants). The choice of rule R2 itself is a reading, not something the pages fix:
"parity unpinned by the pages" for the rule choice, pinned for its execution.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "e2m1_decode", "e8m0_decode", "e4m3fn_decode", "bf16_bits_from_f64", "bf16_bits_to_f64",
    "unpack_nibbles", "mxfp4_values", "mxfp4_dequant", "fp8_block_dequant_128x128",
    "act_quant_mxfp4", "mxfp4_gemm_bf16", "mxfp4_gemm_blockint", "moe_route", "moe_forward",
    "nvfp4_values", "nvfp4_dequant", "nvfp4_gemm_f64", "nvfp4_gemm_bf16",
    "e4m3_round_code", "nvfp4_quantize", "moe_nvfp4_forward", "nvfp4_gemm_segments_bf16",
    "nvfp4_activation_global",
    "act_quant_mxfp8", "mxfp8_values", "moe_mxfp8_forward", "mxfp8_mxfp4_gemm_bf16",
    "moe_flops_per_pair", "moe_l1_exact", "swiglu_bf16", "moe_l2_bf16", "moe_combine",
]

# --------------------------------------------------------------------------------------
# Element formats (OCP MX v1.0 bit fields)
# --------------------------------------------------------------------------------------


def e2m1_decode(code) -> np.ndarray:
    """E2M1 nibble -> float64: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.

    Exponent field 0 is subnormal: (-1)^s * m/2. Otherwise (-1)^s * (1 + m/2) * 2^(e-1).
    Code 0 is +0.0 and code 8 is -0.0 [FMT].
    """
    c = np.asarray(code).astype(np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + 0.5 * m) * np.ldexp(1.0, e - 1))
    return np.where(s == 1, -mag, mag)


def e8m0_decode(b) -> np.ndarray:
    """E8M0 scale byte -> float64: 2^(b - 127); byte 255 is NaN."""
    v = np.asarray(b).astype(np.int64)
    return np.where(v == 255, np.nan, np.ldexp(1.0, v - 127))


def e4m3fn_decode(b) -> np.ndarray:
    """E4M3 ("fn") byte -> float64: sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0.

    Exponent field 0 is subnormal: (-1)^s * (m/8) * 2^-6. S.1111.111 is NaN; no infinity.
    """
    v = np.asarray(b).astype(np.int64)
    s = (v >> 7) & 1
    e = (v >> 3) & 15
    m = v & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def bf16_bits_from_f64(x, nan_sign=None) -> np.ndarray:
    """Round float64 values to BF16 (reading R8) and return uint16 bit patterns.

    The rounding quantum of a finite |x| is 2^(floor(log2|x|) - 7) for |x| >= 2^-126 and
    2^-133 below (BF16 subnormals). Results at or beyond 2^128 are infinite. NaN becomes
    0x7FC0, with the sign bit taken from ``nan_sign`` (bool array) when given (R7).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    ax = np.abs(x)
    nan = np.isnan(ax)
    ax_safe = np.where(nan | np.isinf(ax), 0.0, ax)
    _, e = np.frexp(ax_safe)                      # ax = f * 2^e, f in [0.5, 1)
    q = np.maximum(e - 1 - 7, -133)               # exponent of the BF16 quantum
    r = np.round(np.ldexp(ax_safe, -q))           # np.round: half to even
    mag = np.ldexp(r, q)
    mag = np.where(np.isinf(ax) | (mag >= 2.0 ** 128), np.inf, mag)
    bits = (mag.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = bits | (neg.astype(np.uint16) << 15)
    if nan.any():
        ns = neg if nan_sign is None else np.broadcast_to(np.asarray(nan_sign, dtype=bool), x.shape)
        bits = np.where(nan, (0x7FC0 | (ns.astype(np.uint16) << 15)).astype(np.uint16), bits)
    return bits.astype(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------------------
# MXFP4 tensors [FMT], [DQ] item 2
# --------------------------------------------------------------------------------------


def unpack_nibbles(codes) -> np.ndarray:
    """uint8 [..., C/2] -> nibbles uint8 [..., C]: byte j holds column 2j in its lower
    nibble and column 2j+1 in its upper nibble ("lower nibble first") [DQ] item 2."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (2 * c.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = c & 0x0F
    out[..., 1::2] = c >> 4
    return out


def mxfp4_values(codes, sf) -> np.ndarray:
    """Exact float64 value of an MXFP4 tensor: LUT[code(r, c)] * 2^(sf[r, c // 32] - 127).

    codes uint8 [..., C/2], sf uint8 [..., C/32] -> float64 [..., C] [DQ] item 2.
    """
    nib = unpack_nibbles(codes)
    C = nib.shape[-1]
    sf = np.asarray(sf, dtype=np.uint8)
    if sf.shape[-1] * 32 != C:
        raise ValueError("need one scale per 32 logical columns")
    lut = e2m1_decode(np.arange(16))                 # the 16-entry E2M1 LUT
    scales = e8m0_decode(np.arange(256))             # the 256 E8M0 scale values
    return lut[nib] * np.repeat(scales[sf], 32, axis=-1)


def mxfp4_dequant(codes, sf) -> np.ndarray:
    """MXFP4 -> BF16 bits [R, C] (exact whenever finite). NaN keeps the code's sign (R7)."""
    nib = unpack_nibbles(codes)
    vals = mxfp4_values(codes, sf)
    return bf16_bits_from_f64(vals, nan_sign=(nib >> 3).astype(bool))


def fp8_block_dequant_128x128(q, sf) -> np.ndarray:
    """FP8 E4M3 x E8M0 128x128 block scale -> BF16 bits [R, C] ([DQ] item 1, [DG] item 1).

    out[i, j] = e4m3(q[i, j]) * 2^(sf[i // 128, j // 128] - 127); partial edge blocks use
    the scale of the block they fall in. sf has shape [ceil(R/128), ceil(C/128)].
    """
    q = np.asarray(q, dtype=np.uint8)
    R, C = q.shape
    sf = np.asarray(sf, dtype=np.uint8)
    if sf.shape != ((R + 127) // 128, (C + 127) // 128):
        raise ValueError("scale grid must be [ceil(R/128), ceil(C/128)]")
    s = e8m0_decode(sf)
    scale = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:R, :C]
    vals = e4m3fn_decode(np.arange(256))[q] * scale  # 256-entry E4M3 table, then the block scale
    return bf16_bits_from_f64(vals, nan_sign=(q >> 7).astype(bool))


# --------------------------------------------------------------------------------------
# NVFP4 tensors (readings R11, R12) [NVQ], [GS]
# --------------------------------------------------------------------------------------


def nvfp4_values(codes, sf, global_scale) -> np.ndarray:
    """Exact float64 value of an NVFP4 tensor (R11): LUT[code(r, c)] * e4m3(sf[r, c // 16])
    * global. codes uint8 [..., C/2], sf uint8 [..., C/16] (E4M3 bytes), global a float32
    scalar. Exact: the three factors carry at most 2 + 4 + 24 significant bits."""
    nib = unpack_nibbles(codes)
    C = nib.shape[-1]
    sf = np.asarray(sf, dtype=np.uint8)
    if sf.shape[-1] * 16 != C:
        raise ValueError("need one scale per 16 logical columns")
    lut = e2m1_decode(np.arange(16))
    e4 = e4m3fn_decode(np.arange(256))
    g = float(np.float32(global_scale))
    with np.errstate(invalid="ignore"):
        return lut[nib] * np.repeat(e4[sf], 16, axis=-1) * g


def nvfp4_dequant(codes, sf, global_scale) -> np.ndarray:
    """NVFP4 -> BF16 bits [R, C] (R12): the exact value rounded to float32, then to BF16."""
    nib = unpack_nibbles(codes)
    sf = np.asarray(sf, dtype=np.uint8)
    vals = nvfp4_values(codes, sf, global_scale)
    with np.errstate(over="ignore", invalid="ignore"):
        f32 = vals.astype(np.float32).astype(np.float64)       # IEEE round to nearest even
    g_neg = bool(np.signbit(np.float32(global_scale)))
    sign = ((nib >> 3) ^ np.repeat(sf >> 7, 16, axis=-1) ^ np.uint8(g_neg)).astype(bool)
    return bf16_bits_from_f64(f32, nan_sign=sign)


# --------------------------------------------------------------------------------------
# Activation quantisation (reading R2) [PIPE] "re-quant"
# --------------------------------------------------------------------------------------

_E2M1_MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_round_magnitude(a) -> np.ndarray:
    """Magnitude code 0..7 of the E2M1 value nearest to a >= 0, ties to the even code
    (mantissa bit 0), saturating at 6."""
    a = np.minimum(np.asarray(a, dtype=np.float64), 6.0)
    d = np.abs(a[..., None] - _E2M1_MAGS)                     # distance to each magnitude
    best = d.min(axis=-1, keepdims=True)
    cand = d == best                                           # one, or two on a tie
    idx = np.arange(8)
    even = cand & ((idx & 1) == 0)
    # on a tie the two candidates are adjacent codes, exactly one of them even
    pick = np.where(even.any(axis=-1, keepdims=True), even, cand)
    return np.argmax(pick, axis=-1).astype(np.uint8)


def act_quant_mxfp4(x_bits):
    """BF16 [M, K] -> (codes uint8 [M, K/2], sf uint8 [M, K/32]) by reading R2.

    Per row and per block of 32 columns: amax = max |x|; scale byte
    E = clamp(floor(log2 amax) - 2 + 127, 0, 254) (E = 0 when amax = 0); each element is
    v = x * 2^(127 - E) rounded to E2M1 (nearest, ties to even, saturating at 6) with the
    sign of x kept; lower nibble = even column. Non-finite blocks: E = 255, codes sign|7.
    """
    xb = np.asarray(x_bits, dtype=np.uint16)
    M, K = xb.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    if M > 256:                                   # bound the memory of the rounding search
        parts = [act_quant_mxfp4(xb[i:i + 256]) for i in range(0, M, 256)]
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
    x = bf16_bits_to_f64(xb).reshape(M, K // 32, 32)
    finite = np.isfinite(x).all(axis=-1)
    ax = np.abs(np.where(np.isfinite(x), x, 0.0))
    amax = ax.max(axis=-1)
    _, e = np.frexp(amax)                          # amax = f * 2^e -> floor(log2) = e - 1
    E = np.where(amax > 0, np.clip(e - 1 - 2 + 127, 0, 254), 0).astype(np.int64)
    v = np.abs(x) * np.ldexp(1.0, 127 - E)[..., None]
    mag = _e2m1_round_magnitude(np.where(np.isfinite(v), v, 0.0))
    sign = np.signbit(x).astype(np.uint8)
    code = (sign << 3) | mag
    code = np.where(finite[..., None], code, (sign << 3) | 7).astype(np.uint8)
    sf = np.where(finite, E, 255).astype(np.uint8)
    code = code.reshape(M, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf


# --------------------------------------------------------------------------------------
# NVFP4 quantisation (reading R15) [GS]
# --------------------------------------------------------------------------------------

_E4M3_NONNEG = e4m3fn_decode(np.arange(127))          # codes 0..126, increasing, 0 .. 448


def e4m3_round_code(a) -> np.ndarray:
    """Code 0..126 of the E4M3 value nearest to a (float64, 0 <= a <= 448), ties to the
    even code (the even mantissa)."""
    a = np.asarray(a, dtype=np.float64)
    hi = np.clip(np.searchsorted(_E4M3_NONNEG, a, side="left"), 0, 126)   # first value >= a
    lo = np.clip(hi - 1, 0, 126)
    dlo = a - _E4M3_NONNEG[lo]
    dhi = _E4M3_NONNEG[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    return pick.astype(np.uint8)


def nvfp4_quantize(x_bits, global_scale):
    """BF16 [M, K] -> (codes uint8 [M, K/2], sf uint8 [M, K/16] E4M3) by reading R15, with
    the float32 global scale g (finite, in [2^-117, 2^100] so every step stays normal)."""
    xb = np.asarray(x_bits, dtype=np.uint16)
    M, K = xb.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if M > 256:                                   # bound the memory of the rounding search
        parts = [nvfp4_quantize(xb[i:i + 256], global_scale) for i in range(0, M, 256)]
        return (np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
    f32 = np.float32
    g = f32(global_scale)
    r = f32(1.0) / (f32(6.0) * g)
    x = bf16_bits_to_f64(xb).astype(np.float32).reshape(M, K // 16, 16)   # exact
    finite = np.isfinite(x).all(axis=-1)
    amax = np.abs(np.where(np.isfinite(x), x, f32(0.0))).max(axis=-1)
    with np.errstate(over="ignore"):
        t = np.minimum(amax * r, f32(448.0))                              # float32 product
    S = e4m3_round_code(t.astype(np.float64))
    d = e4m3fn_decode(S).astype(np.float32) * g                           # float32 product
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        rd = f32(1.0) / d                                                 # float32 reciprocal
        v = x * rd[..., None]                                             # float32 products
    mag = _e2m1_round_magnitude(np.where(np.isfinite(v), np.abs(v), 6.0).astype(np.float64))
    mag = np.where((S == 0)[..., None], 0, mag)
    sign = np.signbit(x).astype(np.uint8)
    code = np.where(finite[..., None], (sign << 3) | mag, (sign << 3) | 7).astype(np.uint8)
    sf = np.where(finite, S, 0x7F).astype(np.uint8)
    code = code.reshape(M, K)
    return (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8), sf


def nvfp4_activation_global(batches) -> float:
    """Warm-up calibration of an NVFP4 activation global by reading R19: over every BF16
    batch (uint16 [M, K] each), amax = the largest finite |x|; the global is amax / (6 * 448)
    rounded once to float32 (nearest even), clamped to [2^-117, 2^100] (R15's range).
    6 * 448 is the largest NVFP4 magnitude (E2M1 6 times E4M3 448), so the largest input
    quantises to it without clipping."""
    amax = 0.0
    for xb in batches:
        x = bf16_bits_to_f64(np.asarray(xb, dtype=np.uint16))
        x = np.abs(x[np.isfinite(x)])
        if x.size:
            amax = max(amax, float(x.max()))
    g = np.float32(np.float32(amax) / np.float32(6 * 448))     # one float32 division
    return float(np.clip(g, np.float32(2.0 ** -117), np.float32(2.0 ** 100)))


# --------------------------------------------------------------------------------------
# GEMM over MXFP4 operands [PIPE] (L1 / L2 GEMM; one group is a plain GEMM)
# --------------------------------------------------------------------------------------


def mxfp4_gemm_bf16(a_codes, a_sf, b_codes, b_sf) -> np.ndarray:
    """y = bf16(A . B^T) with A [M, K] and B [N, K] MXFP4 (row-major, K-contiguous, the
    nn.Linear [out, in] layout). The float64 dot product is exact for these inputs."""
    A = mxfp4_values(a_codes, a_sf)
    B = mxfp4_values(b_codes, b_sf)
    return bf16_bits_from_f64(A @ B.T)


def mxfp4_gemm_blockint(a_codes, a_sf, b_codes, b_sf) -> np.ndarray:
    """Second formulation of A . B^T (float64 result, not rounded), used as a cross-check:
    per 32-column block the dot product of the doubled E2M1 values is an integer (at most
    32 * 144 in magnitude), scaled by 2^(sa + sb - 254 - 2); the blocks are then summed."""
    na = unpack_nibbles(a_codes)
    nb = unpack_nibbles(b_codes)
    ia = np.rint(2.0 * e2m1_decode(na)).astype(np.int64)
    ib = np.rint(2.0 * e2m1_decode(nb)).astype(np.int64)
    M, K = ia.shape
    N = ib.shape[0]
    ia = ia.reshape(M, K // 32, 32)
    ib = ib.reshape(N, K // 32, 32)
    blk = np.einsum("mbj,nbj->mnb", ia, ib)                     # exact int64
    sa = np.asarray(a_sf, dtype=np.int64)
    sb = np.asarray(b_sf, dtype=np.int64)
    expo = sa[:, None, :] + sb[None, :, :] - 254 - 2
    terms = np.ldexp(blk.astype(np.float64), expo)
    terms = np.where((sa[:, None, :] == 255) | (sb[None, :, :] == 255), np.nan, terms)
    return terms.sum(axis=-1)


def nvfp4_gemm_f64(a_codes, a_sf, a_global, b_codes, b_sf, b_global) -> np.ndarray:
    """A . B^T for NVFP4 A [M, K] and B [N, K] (R11) in float64:
    a_global * b_global * sum_k (LUT * e4m3)_a (LUT * e4m3)_b. The sum of the scaled E2M1
    products is exact in float64 while the terms span less than ~2^40 (every input here);
    its product with the two globals is then rounded once to float64."""
    A = nvfp4_values(a_codes, a_sf, 1.0)
    B = nvfp4_values(b_codes, b_sf, 1.0)
    with np.errstate(invalid="ignore", over="ignore"):
        return (A @ B.T) * (float(np.float32(a_global)) * float(np.float32(b_global)))


def nvfp4_gemm_bf16(a_codes, a_sf, a_global, b_codes, b_sf, b_global) -> np.ndarray:
    """y = bf16(A . B^T) for NVFP4 operands (R11): nvfp4_gemm_f64 rounded once to BF16
    (the NVFP4 GEMM the pages plan for their attention projections, "Phase 2: CuTeDSL
    Attention Kernel", with one global scale per operand)."""
    return bf16_bits_from_f64(nvfp4_gemm_f64(a_codes, a_sf, a_global, b_codes, b_sf, b_global))


def nvfp4_gemm_segments_bf16(a_codes, a_sf, a_global, b_codes, b_sf, b_globals, seg_rows) -> np.ndarray:
    """Fused projection (R17): B [N, K] is several weight matrices stacked along N, segment s
    holding seg_rows[s] rows with float32 global b_globals[s]; column n of segment s is
    bf16(a_global * b_globals[s] * sum_k A[m, k] B[n, k]), the sum exact (R14)."""
    seg_rows = [int(r) for r in seg_rows]
    if sum(seg_rows) != np.asarray(b_codes).shape[0] or len(seg_rows) != len(b_globals):
        raise ValueError("segments must cover B's rows, one global each")
    S = nvfp4_values(a_codes, a_sf, 1.0) @ nvfp4_values(b_codes, b_sf, 1.0).T
    g = np.repeat([float(np.float32(a_global)) * float(np.float32(gb)) for gb in b_globals], seg_rows)
    with np.errstate(invalid="ignore", over="ignore"):
        return bf16_bits_from_f64(S * g[None, :])


def moe_flops_per_pair(H: int, I: int) -> int:
    """Multiply-adds x 2 for one routed (token, expert) pair: L1 [2I x H] and L2 [H x I]."""
    return 2 * H * 2 * I + 2 * I * H


# --------------------------------------------------------------------------------------
# Routing permutation [PIPE] "routing, topk, scatter"
# --------------------------------------------------------------------------------------


def moe_route(topk_ids, E: int):
    """Stable grouping of the routed (token, slot) pairs by expert.

    Returns (counts int64 [E], offsets int64 [E+1], row_of int64 [T, K] with -1 for
    dropped pairs, tok_of int64 [R]) where the rows of expert e are
    offsets[e] .. offsets[e+1]-1 in (token, slot) order, R = number of valid pairs.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, K = ids.shape
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.nonzero(valid)[0]
    order = order[np.argsort(flat[order], kind="stable")]       # (expert, token, slot)
    row_of = np.full(T * K, -1, dtype=np.int64)
    row_of[order] = np.arange(order.size)
    tok_of = order // K
    return counts, offsets, row_of.reshape(T, K), tok_of


# --------------------------------------------------------------------------------------
# MoE expert FFN [PIPE], [BF16]; readings R1, R3, R4, R5
# --------------------------------------------------------------------------------------


def _silu(z):
    return z / (1.0 + np.exp(-z))


def moe_l1_exact(xq_vals, w13_e, s13_e, I: int):
    """Exact L1 of one expert: (g, u) as float64 [n, I] each, gate = rows [0, I) (R4)."""
    W13 = mxfp4_values(w13_e, s13_e)                     # [2I, H]
    gu = xq_vals @ W13.T                                 # exact
    return gu[:, :I], gu[:, I:]


def swiglu_bf16(g, u):
    """h = bf16( silu(bf16(g)) * bf16(u) ) from exact g, u (R3); BF16 bits [n, I]. A NaN
    h is the positive 0x7FC0 (R20)."""
    gb = bf16_bits_to_f64(bf16_bits_from_f64(g))
    ub = bf16_bits_to_f64(bf16_bits_from_f64(u))
    with np.errstate(over="ignore", invalid="ignore"):
        h = _silu(gb) * ub
    return bf16_bits_from_f64(h, nan_sign=np.zeros(h.shape, dtype=bool))


def moe_l2_bf16(hq, hs, w2_e, s2_e):
    """y = bf16( hq . w2^T ) exactly rounded (R3); BF16 bits [n, H]."""
    W2 = mxfp4_values(w2_e, s2_e)                        # [H, I]
    return bf16_bits_from_f64(mxfp4_values(hq, hs) @ W2.T)


def moe_combine(y_slots, ids, wts, E: int):
    """out[t] = bf16( sum_k w[t, k] * y[t, k] ) over valid slots, float64 sum (R5).

    y_slots float64 [n, K, H] (values of BF16 numbers), ids int [n, K], wts float32 [n, K].
    """
    ids = np.asarray(ids, dtype=np.int64)
    wts = np.asarray(wts, dtype=np.float32).astype(np.float64)
    n, K = ids.shape
    acc = np.zeros((n, y_slots.shape[-1]), dtype=np.float64)
    for k in range(K):                                   # slot order
        live = (ids[:, k] >= 0) & (ids[:, k] < E)
        acc += np.where(live[:, None], wts[:, k:k + 1] * y_slots[:, k], 0.0)
    return bf16_bits_from_f64(acc)


def _expert_ffn(xq_vals, w13_e, s13_e, w2_e, s2_e, I):
    """One expert on a block of rows: returns y as float64 values of BF16 numbers."""
    g, u = moe_l1_exact(xq_vals, w13_e, s13_e, I)
    hq, hs = act_quant_mxfp4(swiglu_bf16(g, u))          # re-quant             (R2)
    return bf16_bits_to_f64(moe_l2_bf16(hq, hs, w2_e, s2_e))


def moe_forward(x_bits, topk_ids, topk_w, w13, s13, w2, s2, I: int, tokens=None):
    """MoE expert FFN output as BF16 bits [len(tokens), H].

    x_bits uint16 [T, H]; topk_ids int32 [T, K] and topk_w float32 [T, K], or both None
    for the shared expert (E = 1, out = y); w13 uint8 [E, 2I, H/2], s13 [E, 2I, H/32];
    w2 uint8 [E, H, I/2], s2 [E, H, I/32]. ``tokens`` selects the rows to compute (all by
    default); every token's output depends only on its own row and routing.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    E = w13.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xq, xs = act_quant_mxfp4(x_bits[tok])                # first quantisation   (R1)
    xv = mxfp4_values(xq, xs)
    if topk_ids is None:
        if E != 1:
            raise ValueError("the unrouted (shared expert) mode needs exactly one expert")
        y = _expert_ffn(xv, w13[0], s13[0], w2[0], s2[0], I)
        return bf16_bits_from_f64(y)
    ids = np.asarray(topk_ids, dtype=np.int64)[tok]
    n, K = ids.shape
    Y = np.zeros((n, K, H), dtype=np.float64)
    for e in range(E):
        sel = np.argwhere(ids == e)                      # (row in sample, slot)
        if sel.size == 0:
            continue
        Y[sel[:, 0], sel[:, 1]] = _expert_ffn(xv[sel[:, 0]], w13[e], s13[e], w2[e], s2[e], I)
    return moe_combine(Y, ids, np.asarray(topk_w, dtype=np.float32)[tok], E)


# --------------------------------------------------------------------------------------
# NVFP4 MoE expert FFN (reading R16) [PIPE], [GS]
# --------------------------------------------------------------------------------------


def _g64(v) -> float:
    return float(np.float32(v))


def moe_nvfp4_forward(x_bits, topk_ids, topk_w, w13, s13, g13, w2, s2, g2, x_global, h_global, I: int,
                      tokens=None):
    """NVFP4 MoE expert FFN output as BF16 bits [len(tokens), H] (R16).

    As moe_forward, with NVFP4 weights: w13 uint8 [E, 2I, H/2] + s13 [E, 2I, H/16] (E4M3)
    and g13 float32 [E, 2] (gate, up globals); w2 uint8 [E, H, I/2] + s2 [E, H, I/16] and
    g2 float32 [E]; x_global and h_global are the float32 globals of the two activation
    quantisations.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    E = w13.shape[0]
    g13 = np.asarray(g13, dtype=np.float32).reshape(E, 2)
    g2 = np.asarray(g2, dtype=np.float32).reshape(E)
    gx, gh = _g64(x_global), _g64(h_global)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xq, xs = nvfp4_quantize(x_bits[tok], x_global)
    xv = nvfp4_values(xq, xs, 1.0)                       # the global goes with the weight's

    def ffn(rows, e):
        gu = xv[rows] @ nvfp4_values(w13[e], s13[e], 1.0).T                 # exact sums
        g = gu[:, :I] * (gx * float(g13[e, 0]))
        u = gu[:, I:] * (gx * float(g13[e, 1]))
        hq, hs = nvfp4_quantize(swiglu_bf16(g, u), h_global)
        y = (nvfp4_values(hq, hs, 1.0) @ nvfp4_values(w2[e], s2[e], 1.0).T) * (gh * float(g2[e]))
        return bf16_bits_to_f64(bf16_bits_from_f64(y))

    if topk_ids is None:
        if E != 1:
            raise ValueError("the unrouted (shared expert) mode needs exactly one expert")
        return bf16_bits_from_f64(ffn(np.arange(tok.size), 0))
    ids = np.asarray(topk_ids, dtype=np.int64)[tok]
    n, K = ids.shape
    Y = np.zeros((n, K, H), dtype=np.float64)
    for e in range(E):
        sel = np.argwhere(ids == e)
        if sel.size == 0:
            continue
        Y[sel[:, 0], sel[:, 1]] = ffn(sel[:, 0], e)
    return moe_combine(Y, ids, np.asarray(topk_w, dtype=np.float32)[tok], E)


# --------------------------------------------------------------------------------------
# MXFP8 activations (reading R18)
# --------------------------------------------------------------------------------------


def act_quant_mxfp8(x_bits):
    """BF16 [M, K] -> (E4M3 codes uint8 [M, K], E8M0 scales uint8 [M, K/32]) by reading R18."""
    xb = np.asarray(x_bits, dtype=np.uint16)
    M, K = xb.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    x = bf16_bits_to_f64(xb).reshape(M, K // 32, 32)
    finite = np.isfinite(x).all(axis=-1)
    amax = np.abs(np.where(np.isfinite(x), x, 0.0)).max(axis=-1)
    _, e = np.frexp(amax)                          # amax = f * 2^e -> floor(log2) = e - 1
    E = np.where(amax > 0, np.clip(e - 1 - 8 + 127, 0, 254), 0).astype(np.int64)
    v = np.abs(np.where(np.isfinite(x), x, 0.0)) * np.ldexp(1.0, 127 - E)[..., None]   # exact
    mag = e4m3_round_code(np.minimum(v, 448.0))
    sign = (np.signbit(x).astype(np.uint8) << 7)
    code = np.where(finite[..., None], sign | mag, sign | 0x7F).astype(np.uint8)
    sf = np.where(finite, E, 255).astype(np.uint8)
    return code.reshape(M, K), sf


def mxfp8_values(codes, sf) -> np.ndarray:
    """Exact float64 value of an MXFP8 tensor: e4m3(code) * 2^(sf[r, c // 32] - 127)."""
    q = np.asarray(codes, dtype=np.uint8)
    sf = np.asarray(sf, dtype=np.uint8)
    if sf.shape[-1] * 32 != q.shape[-1]:
        raise ValueError("need one scale per 32 columns")
    with np.errstate(invalid="ignore"):
        return e4m3fn_decode(np.arange(256))[q] * np.repeat(e8m0_decode(sf), 32, axis=-1)


def mxfp8_mxfp4_gemm_bf16(a_codes, a_sf, b_codes, b_sf) -> np.ndarray:
    """y = bf16(A . B^T) with MXFP8 A [M, K] (E4M3 codes [M, K], E8M0 [M, K/32]) and MXFP4 B
    [N, K] (codes [N, K/2], E8M0 [N, K/32]): the GEMM of the MXFP8-activation path (R18);
    the float64 sum is exact for these inputs and rounded once."""
    return bf16_bits_from_f64(mxfp8_values(a_codes, a_sf) @ mxfp4_values(b_codes, b_sf).T)


def moe_mxfp8_forward(x_bits, topk_ids, topk_w, w13, s13, w2, s2, I: int, tokens=None):
    """MoE expert FFN with MXFP8 activations and the MXFP4 weights (R18); arguments and
    result as moe_forward."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    E = w13.shape[0]
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    xq, xs = act_quant_mxfp8(x_bits[tok])
    xv = mxfp8_values(xq, xs)

    def ffn(rows, e):
        g, u = moe_l1_exact(xv[rows], w13[e], s13[e], I)                   # exact sums
        hq, hs = act_quant_mxfp8(swiglu_bf16(g, u))
        y = mxfp8_values(hq, hs) @ mxfp4_values(w2[e], s2[e]).T
        return bf16_bits_to_f64(bf16_bits_from_f64(y))

    if topk_ids is None:
        if E != 1:
            raise ValueError("the unrouted (shared expert) mode needs exactly one expert")
        return bf16_bits_from_f64(ffn(np.arange(tok.size), 0))
    ids = np.asarray(topk_ids, dtype=np.int64)[tok]
    n, K = ids.shape
    Y = np.zeros((n, K, H), dtype=np.float64)
    for e in range(E):
        sel = np.argwhere(ids == e)
        if sel.size == 0:
            continue
        Y[sel[:, 0], sel[:, 1]] = ffn(sel[:, 0], e)
    return moe_combine(Y, ids, np.asarray(topk_w, dtype=np.float32)[tok], E)
