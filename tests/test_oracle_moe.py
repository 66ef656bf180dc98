"""Pins for the oracle's routing permutation and MoE forward (CPU only).

Pipeline per "Current Bug: vLLM produces empty/garbage output", "Phase 1: CuTeDSL Shared
Expert Kernel" (L1 GEMM -> SiLU -> re-quant -> L2 GEMM; the MoE adds routing, top-k and
scatter; the shared expert is the MoE with one group and no routing) and "Phase 3: Clean
up" (BF16 for the SiLU activation and the final scatter). The forward is pinned by an
exact-rational brute force on tiny inputs and by invariants that catch a swapped gate/up,
a wrong slot/weight pairing, a dropped expert or a token mix-up.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import bf16_bits_from_f64, bf16_bits_to_f64, moe_forward, moe_route
from workloads import make_moe_inputs

GRID = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
        Fraction(4), Fraction(6)]


def _e2m1(n):
    s, e, m = n >> 3, (n >> 1) & 3, n & 1
    mag = Fraction(m, 2) if e == 0 else (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return -mag if s else mag


def _row_values(codes_row, sf_row):
    out = []
    for c in range(2 * len(codes_row)):
        b = int(codes_row[c // 2])
        n = (b & 15) if c % 2 == 0 else (b >> 4)
        out.append(_e2m1(n) * Fraction(2) ** (int(sf_row[c // 32]) - 127))
    return out


def _bf16(q: Fraction) -> Fraction:
    """Nearest BF16 (ties to even) of a finite exact rational in the normal range."""
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
    return (r * quantum) * (1 if q > 0 else -1)


def _quant_block(vals):
    """Brute-force MX quantisation of 32 exact values: returns their dequantised values."""
    amax = max(abs(v) for v in vals)
    if amax == 0:
        return [Fraction(0)] * 32
    e = math.floor(math.log2(amax))
    while Fraction(2) ** e > amax:
        e -= 1
    while Fraction(2) ** (e + 1) <= amax:
        e += 1
    scale = Fraction(2) ** (e - 2)
    out = []
    for v in vals:
        m = min(abs(v) / scale, Fraction(6))
        d = [abs(m - g) for g in GRID]
        best = min(d)
        cands = [i for i in range(8) if d[i] == best]
        i = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
        out.append(GRID[i] * scale * (-1 if v < 0 else 1))
    return out


def _brute_moe(inp):
    T, H, I = inp.T, inp.H, inp.I
    xs = [[Fraction(float(v)) for v in bf16_bits_to_f64(inp.x[t])] for t in range(T)]
    out = []
    for t in range(T):
        xq = sum((_quant_block(xs[t][b:b + 32]) for b in range(0, H, 32)), [])
        acc = Fraction(0)
        accv = [Fraction(0)] * H
        for k in range(inp.K):
            e = int(inp.topk_ids[t, k]) if inp.topk_ids is not None else 0
            if not (0 <= e < inp.w13.shape[0]):
                continue
            wgt = Fraction(float(inp.topk_w[t, k])) if inp.topk_w is not None else Fraction(1)
            W13 = [_row_values(inp.w13[e, r], inp.s13[e, r]) for r in range(2 * I)]
            gu = [sum(a * b for a, b in zip(xq, W13[r])) for r in range(2 * I)]
            g = [_bf16(v) for v in gu[:I]]
            u = [_bf16(v) for v in gu[I:]]
            h = [_bf16(Fraction(float(gg) / (1.0 + math.exp(-float(gg)))) * uu) for gg, uu in zip(g, u)]
            hq = sum((_quant_block(h[b:b + 32]) for b in range(0, I, 32)), [])
            W2 = [_row_values(inp.w2[e, r], inp.s2[e, r]) for r in range(H)]
            y = [_bf16(sum(a * b for a, b in zip(hq, W2[r]))) for r in range(H)]
            accv = [a + wgt * yy for a, yy in zip(accv, y)]
        out.append([float(_bf16(a)) for a in accv])
    return np.array(out)


@pytest.mark.parametrize("routed", [True, False])
def test_moe_brute_force_tiny(routed):
    if routed:
        inp = make_moe_inputs(T=3, H=64, I=32, E=3, K=2, seed=21, routing="uniform",
                              sf_lo=120, sf_hi=126)
    else:
        inp = make_moe_inputs(T=2, H=64, I=32, E=1, K=1, seed=22, routing=None,
                              sf_lo=120, sf_hi=126)
    got = bf16_bits_to_f64(moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13,
                                       inp.w2, inp.s2, inp.I))
    want = _brute_moe(inp)
    # SiLU uses float64 exp in both; everything else is exact -> identical BF16 outputs
    np.testing.assert_array_equal(got, want)


def test_route_invariants():
    rng = np.random.default_rng(4)
    T, K, E = 50, 4, 6
    ids = rng.integers(-2, E + 2, size=(T, K)).astype(np.int32)
    counts, offsets, row_of, tok_of = moe_route(ids, E)
    valid = (ids >= 0) & (ids < E)
    assert counts.sum() == valid.sum()
    assert offsets[0] == 0 and offsets[-1] == valid.sum()
    rows = row_of[valid]
    assert sorted(rows.tolist()) == list(range(valid.sum()))      # each pair exactly once
    assert (row_of[~valid] == -1).all()
    for e in range(E):
        sel = [(t, k) for t in range(T) for k in range(K) if ids[t, k] == e]
        got = [int(row_of[t, k]) for t, k in sel]
        assert got == list(range(offsets[e], offsets[e + 1]))     # stable, grouped by expert
        assert [int(tok_of[r]) for r in got] == [t for t, _ in sel]


def _small(seed, **kw):
    args = dict(T=6, H=64, I=64, E=3, K=2, seed=seed, routing="uniform", sf_lo=120, sf_hi=126)
    args.update(kw)
    return make_moe_inputs(**args)


def _run(inp, ids=None, w=None, **over):
    p = dict(w13=inp.w13, s13=inp.s13, w2=inp.w2, s2=inp.s2)
    p.update(over)
    return moe_forward(inp.x, inp.topk_ids if ids is None else ids,
                       inp.topk_w if w is None else w, p["w13"], p["s13"], p["w2"], p["s2"], inp.I)


def test_shared_mode_equals_single_expert_routing():
    inp = make_moe_inputs(T=5, H=64, I=64, E=1, K=1, seed=31, routing=None)
    shared = moe_forward(inp.x, None, None, inp.w13, inp.s13, inp.w2, inp.s2, inp.I)
    ids = np.zeros((5, 1), np.int32)
    w = np.ones((5, 1), np.float32)
    routed = moe_forward(inp.x, ids, w, inp.w13, inp.s13, inp.w2, inp.s2, inp.I)
    np.testing.assert_array_equal(shared, routed)


def test_dropped_ids_and_zero_up_give_zero():
    inp = _small(32)
    out = _run(inp, ids=np.full_like(inp.topk_ids, -1))
    assert (bf16_bits_to_f64(out) == 0).all()
    w13 = inp.w13.copy()
    w13[:, inp.I:, :] = 0                       # up rows are zero -> h = 0 -> out = 0
    assert (bf16_bits_to_f64(_run(inp, w13=w13)) == 0).all()


def test_gate_is_first_half():
    """A strongly negative gate switches SiLU off; a strongly negative up does not."""
    inp = _small(33, E=1, K=1, routing=None)
    w13 = inp.w13.copy()
    s13 = inp.s13.copy()
    x = bf16_bits_to_f64(inp.x)
    # choose the sign pattern of gate rows so g = -|large| for every token: all weights of a
    # gate row equal -6 where x > 0 and +6 where x < 0 would depend on x; instead use x = 1.
    xb = np.full_like(inp.x, 0x3F80)                                 # x = 1.0 everywhere
    w13[:, :inp.I, :] = 0xFF                                         # gate weights -6
    w13[:, inp.I:, :] = 0x22                                         # up weights +1
    s13[:] = 127
    out_neg_gate = moe_forward(xb, None, None, w13, s13, inp.w2, inp.s2, inp.I)
    w13b = w13.copy()
    w13b[:, :inp.I, :] = 0x22
    w13b[:, inp.I:, :] = 0xFF
    out_neg_up = moe_forward(xb, None, None, w13b, s13, inp.w2, inp.s2, inp.I)
    assert (bf16_bits_to_f64(out_neg_gate) == 0).all()               # silu(-384) ~ 0
    assert np.abs(bf16_bits_to_f64(out_neg_up)).max() > 0


def test_token_independence_and_sampling():
    inp = _small(34, T=9)
    full = _run(inp)
    part = moe_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.w2, inp.s2, inp.I,
                       tokens=[7, 2, 4])
    np.testing.assert_array_equal(part, full[[7, 2, 4]])


def test_expert_relabelling_invariance():
    inp = _small(35)
    perm = np.array([2, 0, 1])                                       # new label of old expert
    inv = np.argsort(perm)
    out = _run(inp, ids=perm[inp.topk_ids].astype(np.int32), w13=inp.w13[inv], s13=inp.s13[inv],
               w2=inp.w2[inv], s2=inp.s2[inv])
    np.testing.assert_array_equal(out, _run(inp))


def test_weight_linearity_and_slot_pairing():
    inp = _small(36)
    out = bf16_bits_to_f64(_run(inp))
    np.testing.assert_array_equal(bf16_bits_to_f64(_run(inp, w=inp.topk_w * 2)), 2 * out)
    # swapping the slots together with their weights changes nothing (only the float64
    # summation order changes, which is exact here up to one final rounding)
    sw = _run(inp, ids=inp.topk_ids[:, ::-1].copy(), w=inp.topk_w[:, ::-1].copy())
    np.testing.assert_allclose(bf16_bits_to_f64(sw), out, rtol=2 ** -8, atol=0)
    # zero weight on slot 1 equals routing slot 1 to nowhere
    w = inp.topk_w.copy()
    w[:, 1] = 0
    ids = inp.topk_ids.copy()
    ids[:, 1] = -1
    np.testing.assert_array_equal(_run(inp, w=w), _run(inp, ids=ids))


def test_nan_in_h_is_positive_and_requantises_to_code_7():
    """Reading R20: every way the SwiGLU step makes a NaN -- a NaN g or u of either sign,
    SiLU(-inf) = -inf / inf, 0 * inf, inf * 0 -- gives h = 0x7FC0 (sign clear), and the MX
    re-quant of a block holding it is scale 255 with code 7 there. Finite and infinite h keep
    their signs (R7 is untouched where the inputs define the sign)."""
    from oracle import act_quant_mxfp4, swiglu_bf16
    nan = np.float64("nan")
    g = np.array([[nan, -nan, -np.inf, 0.0, np.inf, 1.0, np.inf, 2.0, -3.0]])
    u = np.array([[1.0, 1.0, 1.0, np.inf, 0.0, -nan, -1.0, -3.0, 0.5]])
    h = swiglu_bf16(g, u)
    assert (h[0, :6] == 0x7FC0).all()
    assert h[0, 6] == 0xFF80                               # silu(inf) * -1 = -inf
    # silu(2) * -3 and silu(-3) * 0.5: finite, sign of the product, nearest-even BF16
    for i, (gi, ui) in enumerate([(2.0, -3.0), (-3.0, 0.5)], start=7):
        want = bf16_bits_from_f64(gi / (1.0 + math.exp(-gi)) * ui)
        assert h[0, i] == want and (h[0, i] >> 15) == 1
    block = np.concatenate([h[:, :1], np.full((1, 31), bf16_bits_from_f64(np.array(-1.5)), np.uint16)], axis=1)
    q, s = act_quant_mxfp4(block)
    assert s[0, 0] == 255
    assert q[0, 0] & 0x0F == 0x7                           # element 0: the positive NaN
    assert (q[0, 0] >> 4) == 0xF and (q[0, 1:] == 0xFF).all()   # the rest: sign | 7
