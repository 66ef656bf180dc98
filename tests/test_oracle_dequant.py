"""Pins for the oracle's MXFP4 and FP8 128x128 dequantisation (CPU only).

Sources: "2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", sections "Script update:
dequant_fp8_to_bf16.py now handles ALL compressed types" (items 1 and 2: lower nibble
first, one E8M0 scale per row per 32 columns, FP8 x E8M0 per 128x128 block) and "FP4 (E2M1)
expert weight format confirmed" (stored/logical shapes, 224 * 32 = 7168, 96 * 32 = 3072).
Values are checked against torch's float8 conversions and float32 -> bfloat16 rounding.
"""
import json
import os

import numpy as np
import torch

from oracle import bf16_bits_to_f64, fp8_block_dequant_128x128, mxfp4_dequant, mxfp4_values

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FACTS = json.load(open(os.path.join(GOLDEN, "page_facts.json")))


def _torch_bf16_bits(values_f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32)).to(
        torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)


def test_nibble_order_one_hot():
    # byte 0x0F: lower nibble = 15 (-6) is column 0, upper nibble = 0 (+0) is column 1
    codes = np.zeros((1, 16), np.uint8)
    sf = np.full((1, 1), 127, np.uint8)
    codes[0, 0] = 0x0F
    v = mxfp4_values(codes, sf)[0]
    assert v[0] == -6.0 and v[1] == 0.0 and not np.signbit(v[1])
    codes[0, 0] = 0xF0
    v = mxfp4_values(codes, sf)[0]
    assert v[0] == 0.0 and v[1] == -6.0
    codes[0, 0] = 0x21            # column 0 = code 1 (0.5), column 1 = code 2 (1.0)
    v = mxfp4_values(codes, sf)[0]
    assert v[0] == 0.5 and v[1] == 1.0 and (v[2:] == 0).all()


def test_scale_block_indexing():
    rng = np.random.default_rng(1)
    R, C = 3, 128
    codes = rng.integers(0, 256, size=(R, C // 2), dtype=np.uint8)
    sf = np.full((R, C // 32), 127, np.uint8)
    base = mxfp4_dequant(codes, sf)
    for r in range(R):
        for b in range(C // 32):
            s2 = sf.copy()
            s2[r, b] = 129
            got = mxfp4_dequant(codes, s2)
            diff = np.argwhere(bf16_bits_to_f64(got) != bf16_bits_to_f64(base))
            assert diff.size > 0
            assert (diff[:, 0] == r).all()
            assert diff[:, 1].min() >= 32 * b and diff[:, 1].max() < 32 * b + 32
            # inside the block every value is scaled by exactly 4
            blk = slice(32 * b, 32 * b + 32)
            np.testing.assert_array_equal(bf16_bits_to_f64(got)[r, blk], 4 * bf16_bits_to_f64(base)[r, blk])


def test_page_shape_identities():
    sh = FACTS["expert_shapes"]
    for a, b, c in sh["identities"]:
        assert a * b == c
    for name in ("w1", "w3", "w2"):
        stored, scale, logical = sh[name]["stored"], sh[name]["scale"], sh[name]["logical"]
        codes = np.zeros(stored, np.uint8)
        sf = np.full(scale, 127, np.uint8)
        out = mxfp4_dequant(codes, sf)
        assert list(out.shape) == logical
        assert logical[1] == FACTS["nibble_order"]["output_columns_factor"] * stored[1]
        assert scale[1] * FACTS["nibble_order"]["block_columns"] == logical[1]
    ps = FACTS["packed_size"]
    assert round(ps["shape"][0] * ps["shape"][1] / 1e6) == ps["megabytes_rounded"]


def test_all_codes_all_scales_match_torch():
    """Every (code, scale) pair: value = E2M1 x E8M0 via torch's float8/float4-free path."""
    codes = np.arange(256, dtype=np.uint8).reshape(16, 16)          # 16 rows x 32 columns
    for s in range(256):
        sf = np.full((16, 1), s, np.uint8)
        got = mxfp4_dequant(codes, sf)
        # reference: torch e8m0 scale x tabulated e2m1 value, in float32 (exact), then bf16
        e2m1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6], np.float32)
        nib = np.empty((16, 32), np.uint8)
        nib[:, 0::2] = codes & 15
        nib[:, 1::2] = codes >> 4
        scale = torch.tensor([s], dtype=torch.uint8).view(torch.float8_e8m0fnu).float().item()
        with np.errstate(over="ignore", invalid="ignore"):
            ref_f32 = e2m1[nib] * np.float32(scale)
        ref = _torch_bf16_bits(ref_f32)
        if s == 255:
            sign = (nib >> 3).astype(np.uint16)
            assert (got == (0x7FC0 | (sign << 15))).all()
        else:
            np.testing.assert_array_equal(got, ref)


def test_fp8_all_codes_match_torch_and_block_indexing():
    rng = np.random.default_rng(2)
    R, C = 300, 260                                           # ragged edges in both dims
    q = rng.integers(0, 256, size=(R, C), dtype=np.uint8)
    sf = rng.integers(120, 131, size=(3, 3), dtype=np.uint8)
    got = fp8_block_dequant_128x128(q, sf)
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy()
    scale = torch.from_numpy(sf).view(torch.float8_e8m0fnu).float().numpy()
    full = np.repeat(np.repeat(scale, 128, 0), 128, 1)[:R, :C]
    ref = _torch_bf16_bits(vals * full)
    nan = np.isnan(vals)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    sign = (q[nan] >> 7).astype(np.uint16)
    assert (got[nan] == (0x7FC0 | (sign << 15))).all()
    # one-hot scale: a change of block (1, 2) touches rows 128..255 and columns 256..259 only
    s2 = sf.copy()
    s2[1, 2] += 1
    d = np.argwhere(fp8_block_dequant_128x128(q, s2) != got)
    assert d[:, 0].min() >= 128 and d[:, 0].max() <= 255
    assert d[:, 1].min() >= 256 and d[:, 1].max() <= 259


def test_fp8_multiplies_by_block_scale():
    q = np.full((128, 128), 0x38, np.uint8)                    # e4m3 0x38 = 1.0
    sf = np.full((1, 1), 130, np.uint8)                       # 2^3
    out = bf16_bits_to_f64(fp8_block_dequant_128x128(q, sf))
    assert (out == 8.0).all()
