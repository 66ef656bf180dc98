"""Pins for the oracle's element decoders and BF16 rounding (CPU only).

Each check compares the oracle with something other than itself: the OCP MX E2M1 table,
torch's float8 conversions (a library routine), exact rational arithmetic, or facts the
pages print ("2026-05-08 DeepSeek V4 Pro NVFP4 Quantization", "FP4 (E2M1) expert weight
format confirmed": code 0 is +0.0 and code 8 is -0.0).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import bf16_bits_from_f64, bf16_bits_to_f64, e2m1_decode, e4m3fn_decode, e8m0_decode

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, b = line.split()
                rows.append((a, b))
    return rows


def test_e2m1_matches_ocp_table():
    for code, val in _read_table("e2m1_ocp_mx_table.txt"):
        got = float(e2m1_decode(int(code)))
        want = float(val)
        assert got == want, (code, got, want)
        assert math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e2m1_signed_zeros_from_pages():
    facts = json.load(open(os.path.join(GOLDEN, "page_facts.json")))["zero_codes"]
    pz = float(e2m1_decode(facts["plus_zero_code"]))
    mz = float(e2m1_decode(facts["minus_zero_code"]))
    assert pz == 0.0 and not math.copysign(1.0, pz) < 0
    assert mz == 0.0 and math.copysign(1.0, mz) < 0
    assert float(np.max(np.abs(e2m1_decode(np.arange(16))))) == 6.0


def test_e8m0_matches_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = e8m0_decode(np.arange(256))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    np.testing.assert_array_equal(got[:255], ref[:255])
    assert got[127] == 1.0 and got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127


def test_e4m3fn_matches_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3fn_decode(np.arange(256))
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == 448.0
    assert math.copysign(1.0, float(got[0x80])) < 0


def test_bf16_rounding_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(123)
    u = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # add exact ties and values around the overflow threshold and the subnormal range
    extra = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.3895314e38,
                      3.3961776e38, 2.0 ** -130 * 1.5, 2.0 ** -134, 2.0 ** -133 * 1.5, 0.0, -0.0],
                     dtype=np.float32)
    f = np.concatenate([f, extra])
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.uint16).numpy().astype(np.uint16)
    got = bf16_bits_from_f64(f.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_rounding_exact_from_double():
    """Double inputs that are not float32 values: compare with exact rational rounding."""
    rng = np.random.default_rng(7)
    xs = []
    for _ in range(3000):
        e = int(rng.integers(-140, 129))
        m = int(rng.integers(0, 2 ** 52))
        xs.append(math.ldexp(1.0 + m / 2.0 ** 52, e) * (1 if rng.random() < 0.5 else -1))
    # exact ties in double that a float32 detour would break (double rounding)
    xs += [1.0 + 2.0 ** -8 + 2.0 ** -30, 1.0 + 2.0 ** -8 - 2.0 ** -40, 1.0 + 2.0 ** -8]
    got = bf16_bits_from_f64(np.array(xs))
    for x, g in zip(xs, got):
        fx = Fraction(x)
        ax = abs(fx)
        if ax == 0:
            continue
        # quantum from the exact exponent
        e = math.floor(math.log2(abs(x)))
        if Fraction(2) ** e > ax:
            e -= 1
        if Fraction(2) ** (e + 1) <= ax:
            e += 1
        q = Fraction(2) ** max(e - 7, -133)
        n = ax / q
        fl = math.floor(n)
        rem = n - fl
        r = fl + 1 if (rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1)) else fl
        want = r * q
        if want >= Fraction(2) ** 128:
            wv = math.inf
        else:
            wv = float(want)
        wv = -wv if x < 0 else wv
        assert float(bf16_bits_to_f64(g)) == wv, (x, float(bf16_bits_to_f64(g)), wv)


def test_bf16_nan_sign_rule():
    bits = bf16_bits_from_f64(np.array([np.nan, np.nan]), nan_sign=np.array([False, True]))
    assert bits.tolist() == [0x7FC0, 0xFFC0]
    assert bf16_bits_from_f64(np.array([np.inf, -np.inf, 2.0 ** 128])).tolist() == [0x7F80, 0xFF80, 0x7F80]
