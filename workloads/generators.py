"""Seeded input generators (numpy PCG64) for every workload the tests and bench use.

The shapes follow the DeepSeek-V4 expert dimensions printed on the pages:
"2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", section "FP4 (E2M1) expert weight
format confirmed" (w1/w3 stored [3072, 3584] with E8M0 [3072, 224]; w2 stored
[7168, 1536] with E8M0 [7168, 96]), and "Current Bug: vLLM produces empty/garbage
output", section "Config values" (384 routed experts, 48 per expert-parallel rank).

Recipes (one seed per workload; "N(0, s)" means standard deviation s; an E8M0 range
[a, b] means the integers a..b inclusive):

* tiny     seed 0: T=16, H=256, I=128, E=4, top-2; x ~ N(0,1); weight bytes uniform;
                   E8M0 uniform [120, 126]; ids: 2 distinct experts uniform per token;
                   weights = softmax of N(0,1) logits over the chosen experts.
* shared   seed 1: T=256, H=7168, I=3072, one expert, no routing; x ~ N(0,1);
                   weight bytes uniform; E8M0 uniform [118, 124].
* decode   seed 2: T=64, E=48, top-8; router logits N(0,1) [T, 48]; ids = the 8 largest
                   logits (lower expert index first on ties); weights = softmax over the
                   8 chosen logits; x ~ N(0,1); weights as "shared" for every expert.
* prefill  seed 3: T=8192, E=48, top-8; expert probability proportional to 1/rank under
                   a seeded permutation of the experts (Zipf, s = 1); 8 distinct experts
                   per token by Gumbel-top-k over log p; weights = softmax of N(0,1)
                   logits over those 8; x ~ N(0, 0.5) with each element multiplied by 20
                   with probability 0.001.
* dequant  seed 4: MXFP4 weights of 48 experts (w13 [6144, 3584] + [6144, 224] and w2
                   [7168, 1536] + [7168, 96]), E8M0 uniform [118, 124]; FP8 E4M3
                   [7168, 7168] uniform over the 254 finite codes with E8M0 128x128 block
                   scales [56, 56] uniform [120, 130].
* NVFP4 MoE (make_nvfp4_moe_inputs; each MoE config above with its own seed, shapes, x
                   and routing): weight bytes uniform; E4M3 scale bytes uniform over
                   [0x68, 0x7E] (64 .. 448, the top of the range a per-block amax / 6
                   scale fills); weight globals 2^-14 * U[1, 2) * sqrt(7168 / H) for gate
                   and up (drawn separately) and 2^-14 * U[1, 2) * sqrt(3072 / I) for w2,
                   so the L1 sums have the same spread at every size; the x global is the
                   warm-up calibration max|x| / (6 * 448) of the batch itself, the h global
                   the fixed constant 2^-2.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

CONFIGS = {
    "tiny": dict(T=16, H=256, I=128, E=4, K=2, seed=0, routing="uniform",
                 x_sigma=1.0, outlier_p=0.0, sf_lo=120, sf_hi=126),
    "shared": dict(T=256, H=7168, I=3072, E=1, K=1, seed=1, routing=None,
                   x_sigma=1.0, outlier_p=0.0, sf_lo=118, sf_hi=124),
    "decode": dict(T=64, H=7168, I=3072, E=48, K=8, seed=2, routing="topk_logits",
                   x_sigma=1.0, outlier_p=0.0, sf_lo=118, sf_hi=124),
    "prefill": dict(T=8192, H=7168, I=3072, E=48, K=8, seed=3, routing="zipf",
                    x_sigma=0.5, outlier_p=0.001, sf_lo=118, sf_hi=124),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 draws to bfloat16 (nearest, ties to even) and return the bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = (u >> 16) & 1                      # finite values never overflow 32 bits below
    r += 0x7FFF
    r += u
    r >>= 16
    out = r.astype(np.uint16)
    out[np.isnan(x)] = 0x7FC0
    return out


def _uniform_bytes(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform bytes: the generator's raw 64-bit outputs, little-endian, 8 bytes each."""
    n = int(np.prod(shape))
    raw = rng.bit_generator.random_raw((n + 7) // 8).astype("<u8", copy=False)
    return raw.view(np.uint8)[:n].reshape(shape)


def _softmax_f32(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    return (p / p.sum(axis=-1, keepdims=True)).astype(np.float32)


@dataclass
class MoEInputs:
    T: int
    H: int
    I: int
    E: int
    K: int
    x: np.ndarray                      # uint16 bf16 bits [T, H]
    topk_ids: Optional[np.ndarray]     # int32 [T, K] or None (shared expert)
    topk_w: Optional[np.ndarray]       # float32 [T, K] or None
    w13: np.ndarray                    # uint8 [E, 2I, H/2]  rows [0, I) gate, [I, 2I) up
    s13: np.ndarray                    # uint8 [E, 2I, H/32]
    w2: np.ndarray                     # uint8 [E, H, I/2]
    s2: np.ndarray                     # uint8 [E, H, I/32]


def make_routing(rng, T, E, K, routing):
    if routing is None:
        return None, None
    if routing == "uniform":
        ids = np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)]).astype(np.int32)
        w = _softmax_f32(rng.standard_normal((T, K)))
        return ids, w
    if routing == "topk_logits":
        logits = rng.standard_normal((T, E))
        ids = np.argsort(-logits, axis=1, kind="stable")[:, :K].astype(np.int32)
        w = _softmax_f32(np.take_along_axis(logits, ids.astype(np.int64), axis=1))
        return ids, w
    if routing == "zipf":
        perm = rng.permutation(E)
        p = np.empty(E, dtype=np.float64)
        p[perm] = 1.0 / np.arange(1, E + 1)
        p /= p.sum()
        keys = np.log(p)[None, :] + rng.gumbel(size=(T, E))
        ids = np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)
        w = _softmax_f32(rng.standard_normal((T, K)))
        return ids, w
    raise ValueError(f"unknown routing {routing!r}")


def make_moe_inputs(T, H, I, E, K, seed, routing="uniform", x_sigma=1.0, outlier_p=0.0,
                    outlier_scale=20.0, sf_lo=118, sf_hi=124) -> MoEInputs:
    """Draw one MoE workload. ``routing`` is None for the shared expert (E must be 1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((T, H), dtype=np.float32) * np.float32(x_sigma)
    if outlier_p > 0.0:
        mask = rng.random((T, H)) < outlier_p
        x[mask] *= np.float32(outlier_scale)
    ids, w = make_routing(rng, T, E, K, routing)
    w13 = _uniform_bytes(rng, (E, 2 * I, H // 2))
    s13 = rng.integers(sf_lo, sf_hi + 1, size=(E, 2 * I, H // 32), dtype=np.uint8)
    w2 = _uniform_bytes(rng, (E, H, I // 2))
    s2 = rng.integers(sf_lo, sf_hi + 1, size=(E, H, I // 32), dtype=np.uint8)
    return MoEInputs(T, H, I, E, (K if routing is not None else 1), f32_to_bf16_bits(x),
                     ids, w, w13, s13, w2, s2)


def make_config_inputs(name: str) -> MoEInputs:
    c = dict(CONFIGS[name])
    return make_moe_inputs(c.pop("T"), c.pop("H"), c.pop("I"), c.pop("E"), c.pop("K"),
                           c.pop("seed"), **c)


def make_nvfp4_scales(seed=5, experts=48, I=3072, H=7168, lo=0x20, hi=0x5E, global_scale=0.000372):
    """NVFP4 scales for the dequant sweep's expert weights (the codes of make_dequant_inputs):
    E4M3 bytes, one per 16 columns, uniform over the finite positive codes [lo, hi]
    (2^-4 .. 240), and one float32 global scale. Returns (w13 scales [E*2I, H/16],
    w2 scales [E*H, I/16], global)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s13 = rng.integers(lo, hi + 1, size=(experts * 2 * I, H // 16), dtype=np.uint8)
    s2 = rng.integers(lo, hi + 1, size=(experts * H, I // 16), dtype=np.uint8)
    return s13, s2, float(np.float32(global_scale))


def make_gemm_inputs(seed=6, M=8192, N=6144, K=7168):
    """One dense block-scaled GEMM in both formats: uniform code bytes for A [M, K/2] and
    B [N, K/2]; MXFP4 E8M0 scales uniform over [118, 124] per 32 columns; NVFP4 E4M3 scales
    uniform over the positive codes [0x28, 0x48] per 16 columns and float32 globals.
    Returns (a, b, mx_sa, mx_sb, nv_sa, nv_sb, a_global, b_global)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = _uniform_bytes(rng, (M, K // 2))
    b = _uniform_bytes(rng, (N, K // 2))
    mx_sa = rng.integers(118, 125, size=(M, K // 32), dtype=np.uint8)
    mx_sb = rng.integers(118, 125, size=(N, K // 32), dtype=np.uint8)
    nv_sa = rng.integers(0x28, 0x49, size=(M, K // 16), dtype=np.uint8)
    nv_sb = rng.integers(0x28, 0x49, size=(N, K // 16), dtype=np.uint8)
    return a, b, mx_sa, mx_sb, nv_sa, nv_sb, float(np.float32(0.0123)), float(np.float32(0.0457))


def make_dequant_inputs(seed=4, experts=48, I=3072, H=7168, fp8_rows=7168, fp8_cols=7168,
                        sf_lo=118, sf_hi=124, fp8_sf_lo=120, fp8_sf_hi=130):
    """Weight dequant sweep: MXFP4 expert weights flattened to rows, plus one FP8 matrix.

    Returns (mx_codes [R, C/2], mx_sf [R, C/32], w2_codes, w2_sf, fp8_q, fp8_sf) where the
    w13 rows of all experts are flattened into R = experts * 2I rows of C = H columns and
    the w2 rows into experts * H rows of I columns.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    w13 = _uniform_bytes(rng, (experts * 2 * I, H // 2))
    s13 = rng.integers(sf_lo, sf_hi + 1, size=(experts * 2 * I, H // 32), dtype=np.uint8)
    w2 = _uniform_bytes(rng, (experts * H, I // 2))
    s2 = rng.integers(sf_lo, sf_hi + 1, size=(experts * H, I // 32), dtype=np.uint8)
    r = rng.integers(0, 254, size=(fp8_rows, fp8_cols), dtype=np.uint8)
    q = (r + (r >= 127)).astype(np.uint8)          # skip the NaN codes 0x7F and 0xFF
    fsf = rng.integers(fp8_sf_lo, fp8_sf_hi + 1,
                       size=((fp8_rows + 127) // 128, (fp8_cols + 127) // 128), dtype=np.uint8)
    return w13, s13, w2, s2, q, fsf


@dataclass
class NvMoEInputs:
    T: int
    H: int
    I: int
    E: int
    K: int
    x: np.ndarray                      # uint16 bf16 bits [T, H]
    topk_ids: Optional[np.ndarray]     # int32 [T, K] or None (shared expert)
    topk_w: Optional[np.ndarray]       # float32 [T, K] or None
    w13: np.ndarray                    # uint8 [E, 2I, H/2]  rows [0, I) gate, [I, 2I) up
    s13: np.ndarray                    # uint8 [E, 2I, H/16] E4M3
    g13: np.ndarray                    # float32 [E, 2] gate, up globals
    w2: np.ndarray                     # uint8 [E, H, I/2]
    s2: np.ndarray                     # uint8 [E, H, I/16] E4M3
    g2: np.ndarray                     # float32 [E]
    x_global: float                    # float32 values
    h_global: float


NV_H_GLOBAL = 0.25


def make_nvfp4_moe_inputs(T, H, I, E, K, seed, routing="uniform", x_sigma=1.0, outlier_p=0.0,
                          outlier_scale=20.0, sf_lo=0x68, sf_hi=0x7E, h_global=NV_H_GLOBAL, **_unused):
    """Draw one NVFP4 MoE workload (recipe in the module docstring). Accepts the keyword
    arguments of an MXFP4 config (its E8M0 range is ignored)."""
    rng = np.random.Generator(np.random.PCG64(seed + 100))
    x = rng.standard_normal((T, H), dtype=np.float32) * np.float32(x_sigma)
    if outlier_p > 0.0:
        mask = rng.random((T, H)) < outlier_p
        x[mask] *= np.float32(outlier_scale)
    xb = f32_to_bf16_bits(x)
    ids, w = make_routing(rng, T, E, K, routing)
    w13 = _uniform_bytes(rng, (E, 2 * I, H // 2))
    s13 = rng.integers(sf_lo, sf_hi + 1, size=(E, 2 * I, H // 16), dtype=np.uint8)
    w2 = _uniform_bytes(rng, (E, H, I // 2))
    s2 = rng.integers(sf_lo, sf_hi + 1, size=(E, H, I // 16), dtype=np.uint8)
    g13 = (2.0 ** -14 * rng.uniform(1.0, 2.0, size=(E, 2)) * np.sqrt(7168.0 / H)).astype(np.float32)
    g2 = (2.0 ** -14 * rng.uniform(1.0, 2.0, size=E) * np.sqrt(3072.0 / I)).astype(np.float32)
    xv = (xb.astype(np.uint32) << 16).view(np.float32)
    amax = float(np.abs(xv).max()) if T > 0 else 1.0
    x_global = float(np.float32(np.float32(amax) / np.float32(6 * 448)))
    return NvMoEInputs(T, H, I, E, (K if routing is not None else 1), xb, ids, w, w13, s13, g13,
                       w2, s2, g2, x_global, float(np.float32(h_global)))


def make_nvfp4_config_inputs(name: str) -> NvMoEInputs:
    c = dict(CONFIGS[name])
    return make_nvfp4_moe_inputs(c.pop("T"), c.pop("H"), c.pop("I"), c.pop("E"), c.pop("K"),
                                 c.pop("seed"), **c)
