"""Step-by-step parity of a moe_mxfp4_forward (or moe_nvfp4_forward) run against the oracle.

The forward leaves its intermediates in the workspace (moe_mxfp4_workspace_layout), so
every step is checked where it happens:

1. the first MX quantisation of x (xq, xs): bit-exact;
2. the re-quantisation of h = bf16(silu(g) * u): the GPU accumulates g and u in float32,
   the oracle exactly, so an h that sits within that rounding of a BF16 or E2M1 decision
   boundary may legitimately land on either side. Each GPU block (scale + 32 codes) must be
   the MX quantisation of some h' whose elements lie in the interval that the float32
   accumulation allowance and float32 SiLU allow around the oracle's h (decisions that
   the oracle pins uniquely must match exactly). The number of blocks whose decision
   differs from the oracle's own is bounded too: at most FLIP_FRAC of all blocks (never
   less than FLIP_MIN), so a systematic drift that stays inside every block's window
   (a biased SiLU, a lossy accumulation) still fails;
3. y (L2, BF16): within one BF16 rounding plus the float32 accumulation allowance of the
   exact product of the GPU's own hq with w2;
4. out: per element |err| <= 2e-2 * max|ref| + 1e-3 and cosine >= 0.9999 against the
   oracle run on the same decisions (the GPU's hq); against the unconditioned oracle,
   cosine >= 0.9999 over the sample and the same per-element bound on every token whose
   re-quant decisions all equal the oracle's (a token with a flipped block legitimately
   differs by a whole E2M1 step of h times a column of w2).
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle.mxfp4_oracle import _e2m1_round_magnitude
from gpu_util import (MOE_ABS, MOE_COS, MOE_REL, assert_gemm_close, assert_moe_close, bf16_host, bits_to_f64,
                      cosine)

ACC_ALLOW = 2.0 ** -14      # float32 accumulation allowance, relative to sum |a||b|
SILU_ALLOW = 2.0 ** -20     # float32 SiLU / product allowance, relative
# Re-quant blocks allowed to differ from the oracle's decision (step 2). A block differs
# only where the float32 accumulation or SiLU moves one of its BF16 or E2M1 decisions
# across a boundary; measured on the full-size shared, decode and prefill configs with
# E2M1 codes (MXFP4 and NVFP4) that is 1.6e-4 to 6e-4 of the blocks. The cap is 2^-9
# (about 2e-3), three to twelve times that, with a floor of 4 blocks for small samples.
# E4M3 codes (MXFP8 activations, reading R18) carry 3 mantissa bits against E2M1's 1, so
# their decision boundaries are 4x denser and a one-ULP change of h moves a code 4x as
# often: the cap scales by that factor to 2^-7 (measured 6.7e-4 to 2.2e-3).
FLIP_FRAC = 2.0 ** -9
FLIP_FRAC_E4M3 = FLIP_FRAC * 4
FLIP_MIN = 4


def flip_cap(blocks: int, frac: float = FLIP_FRAC) -> int:
    return max(FLIP_MIN, int(frac * blocks))


def check_mx8_requant_decisions(g, u, absg, absu, hq_gpu, hs_gpu):
    """Step 2 for MXFP8 activations (reading R18): every GPU block (E8M0 scale + 32 E4M3
    codes) must be the MXFP8 quantisation of some h' in the interval the float32
    accumulation and SiLU allow around the oracle's h. Returns (differ [n, I/32], at_risk)
    as check_requant_decisions."""
    n, I = g.shape
    h_lo, h_hi = _h_interval(g, u, absg, absu)
    mag_lo = np.where((h_lo <= 0) & (h_hi >= 0), 0.0, np.minimum(np.abs(h_lo), np.abs(h_hi)))
    mag_hi = np.maximum(np.abs(h_lo), np.abs(h_hi))
    nb = I // 32

    def scale_byte(amax):
        _, e = np.frexp(amax)
        return np.where(amax > 0, np.clip(e - 1 - 8 + 127, 0, 254), 0)

    E_lo = scale_byte(mag_lo.reshape(n, nb, 32).max(-1))
    E_hi = scale_byte(mag_hi.reshape(n, nb, 32).max(-1))
    hs = hs_gpu.astype(np.int64)
    bad_scale = (hs < E_lo) | (hs > E_hi) | (hs == 255)
    assert not bad_scale.any(), (f"MXFP8 re-quant scale outside the admissible range at "
                                 f"{np.argwhere(bad_scale)[0].tolist()}")
    mult = np.repeat(np.ldexp(1.0, 127 - hs), 32, axis=1)
    table = oracle.e4m3fn_decode(np.arange(256))
    v_gpu = table[hq_gpu]

    def qv(h):
        sv = h * mult
        mag = oracle.e4m3_round_code(np.minimum(np.abs(sv), 448.0))
        return np.where(np.signbit(sv), -1.0, 1.0) * table[mag]

    v_lo, v_hi = qv(h_lo), qv(h_hi)
    bad = (v_gpu < np.minimum(v_lo, v_hi)) | (v_gpu > np.maximum(v_lo, v_hi))
    assert not bad.any(), (f"MXFP8 re-quant code outside the admissible range at {np.argwhere(bad)[0].tolist()}: "
                           f"gpu {v_gpu[bad][0]}, admissible [{v_lo[bad][0]}, {v_hi[bad][0]}]")
    ref_q, ref_s = oracle.act_quant_mxfp8(oracle.swiglu_bf16(g, u))
    differ = (ref_s != hs_gpu) | (ref_q.reshape(n, nb, 32) != hq_gpu.reshape(n, nb, 32)).any(-1)
    at_risk = (E_lo != E_hi) | (v_lo != v_hi).reshape(n, nb, 32).any(-1)
    return differ, int(at_risk.sum())


def _h_interval(g, u, absg, absu):
    """The extreme BF16 candidates of h = bf16(silu(bf16(g')) * bf16(u')) for g', u' within the
    float32 accumulation allowance of the exact g, u, with the float32 SiLU allowance."""
    to = oracle.bf16_bits_to_f64
    fr = oracle.bf16_bits_from_f64
    eg, eu = absg * ACC_ALLOW, absu * ACC_ALLOW
    gs = [to(fr(g - eg)), to(fr(g + eg))]
    us = [to(fr(u - eu)), to(fr(u + eu))]
    with np.errstate(over="ignore"):
        corners = np.stack([gg / (1.0 + np.exp(-gg)) * uu for gg in gs for uu in us])
    lo = corners.min(0)
    hi = corners.max(0)
    lo = lo - np.abs(lo) * SILU_ALLOW
    hi = hi + np.abs(hi) * SILU_ALLOW
    return to(fr(lo)), to(fr(hi))


def tile_edge_tokens(topk_ids, E: int, tail_tiles: int = 2, per_tail: int = 4, tile_rows: int = 128):
    """A token sample for the large routed configs chosen where grouped-GEMM indexing bugs
    would show: for every expert, the tokens of its first row, of the first row of its last
    128-row M tile and of its last row (the ragged end), plus per_tail tokens spread over each
    of the last tail_tiles M tiles of the grouped order (the work units the persistent GEMM
    grid takes last). The routing comes from the oracle's permutation, which the routing
    tests pin bit-exactly to the GPU's."""
    counts, offsets, _, tok_of = oracle.moe_route(topk_ids, E)
    pick = set()
    tiles = []
    for e in range(E):
        n = int(counts[e])
        if n == 0:
            continue
        o = int(offsets[e])
        last_tile0 = o + ((n - 1) // tile_rows) * tile_rows
        pick.update(int(tok_of[r]) for r in (o, last_tile0, o + n - 1))
        tiles += [(o + m * tile_rows, min(tile_rows, n - m * tile_rows)) for m in range((n + tile_rows - 1) // tile_rows)]
    for r0, n in tiles[-tail_tiles:]:
        pick.update(int(tok_of[r]) for r in np.linspace(r0, r0 + n - 1, per_tail).astype(np.int64))
    return np.array(sorted(pick), dtype=np.int64)


def _ws_scales_stage_major(ws, L, off, R, cols, routed, E, T, block=32):
    """A routed forward's x or h scales (cols = H or I) from the workspace's stage-major layout,
    as row-major [R, cols/block]: per M tile (128 rows of one expert), K stage (256 columns) and
    scale word (4 blocks), the tile's 128 rows' words in row order. block 32: MXFP4 (2 words
    per stage); 16: NVFP4 (4 words per stage)."""
    words = 256 // block // 4
    if routed:
        counts = _ws_view(ws, L["counts"], 1, E, "i32")[0].astype(np.int64)
        offsets = _ws_view(ws, L["offsets"], 1, E + 1, "i32")[0].astype(np.int64)
    else:
        counts, offsets = np.array([T], np.int64), np.array([0, T], np.int64)
    ntiles = (counts + 127) // 128
    tile_base = np.concatenate([[0], np.cumsum(ntiles)])
    k_tiles = -(-cols // 256)
    raw = _ws_view(ws, off, 1, int(tile_base[-1]) * k_tiles * words * 512)[0]
    mt, r = np.zeros(R, np.int64), np.zeros(R, np.int64)
    for e in range(counts.size):
        i = np.arange(counts[e])
        mt[offsets[e] + i] = tile_base[e] + i // 128
        r[offsets[e] + i] = i % 128
    b = np.arange(cols // block)
    byte = (((mt[:, None] * k_tiles + b[None, :] // (4 * words)) * words + (b[None, :] // 4) % words) * 128
            + r[:, None]) * 4 + b[None, :] % 4
    return raw[byte]


def _ws_view(ws, off, rows, cols, dtype=None):
    import torch
    t = ws[off: off + rows * cols * (2 if dtype == "bf16" else 4 if dtype == "i32" else 1)]
    if dtype == "bf16":
        return t.view(torch.int16).view(rows, cols).cpu().numpy().view(np.uint16)
    if dtype == "i32":
        return t.view(torch.int32).view(rows, cols).cpu().numpy()
    return t.view(rows, cols).cpu().numpy()


def _signed_code_value(mag_code, neg):
    return np.where(neg, -1.0, 1.0) * oracle.e2m1_decode(mag_code.astype(np.int64))


def check_requant_decisions(g, u, absg, absu, hq_gpu, hs_gpu):
    """Step 2. Returns (differ [n, I/32]: the block's decision differs from the oracle's own,
    at_risk: blocks whose admissible window holds more than one outcome)."""
    n, I = g.shape
    to = oracle.bf16_bits_to_f64
    fr = oracle.bf16_bits_from_f64
    eg, eu = absg * ACC_ALLOW, absu * ACC_ALLOW
    gs = [to(fr(g - eg)), to(fr(g + eg))]
    us = [to(fr(u - eu)), to(fr(u + eu))]
    with np.errstate(over="ignore"):
        corners = np.stack([gg / (1.0 + np.exp(-gg)) * uu for gg in gs for uu in us])
    lo = corners.min(0)
    hi = corners.max(0)
    lo = lo - np.abs(lo) * SILU_ALLOW
    hi = hi + np.abs(hi) * SILU_ALLOW
    h_lo, h_hi = to(fr(lo)), to(fr(hi))                 # extreme BF16 candidates of h
    # scale byte range over the candidates
    mag_lo = np.where((h_lo <= 0) & (h_hi >= 0), 0.0, np.minimum(np.abs(h_lo), np.abs(h_hi)))
    mag_hi = np.maximum(np.abs(h_lo), np.abs(h_hi))
    nb = I // 32

    def scale_byte(amax):
        _, e = np.frexp(amax)
        return np.where(amax > 0, np.clip(e - 1 - 2 + 127, 0, 254), 0)

    E_lo = scale_byte(mag_lo.reshape(n, nb, 32).max(-1))
    E_hi = scale_byte(mag_hi.reshape(n, nb, 32).max(-1))
    hs = hs_gpu.astype(np.int64)
    bad_scale = (hs < E_lo) | (hs > E_hi) | (hs == 255)
    assert not bad_scale.any(), (f"re-quant scale outside the admissible range at "
                                 f"{np.argwhere(bad_scale)[0].tolist()}")
    mult = np.repeat(np.ldexp(1.0, 127 - hs), 32, axis=1)
    nib = oracle.unpack_nibbles(hq_gpu)
    v_gpu = _signed_code_value(nib & 7, (nib >> 3).astype(bool))

    def qv(h):
        s = h * mult
        return _signed_code_value(_e2m1_round_magnitude(np.minimum(np.abs(s), 6.0)), np.signbit(s))

    v_lo, v_hi = qv(h_lo), qv(h_hi)
    bad = (v_gpu < np.minimum(v_lo, v_hi)) | (v_gpu > np.maximum(v_lo, v_hi))
    assert not bad.any(), (f"re-quant code outside the admissible range at {np.argwhere(bad)[0].tolist()}: "
                           f"gpu {v_gpu[bad][0]}, admissible [{v_lo[bad][0]}, {v_hi[bad][0]}]")
    ref_q, ref_s = oracle.act_quant_mxfp4(oracle.swiglu_bf16(g, u))
    differ = (ref_s != hs_gpu) | (oracle.unpack_nibbles(ref_q).reshape(n, nb, 32) !=
                                  nib.reshape(n, nb, 32)).any(-1)
    at_risk = (E_lo != E_hi) | (v_lo != v_hi).reshape(n, nb, 32).any(-1)
    return differ, int(at_risk.sum())


def check_moe_run(mx, d, tokens=None, mxfp8=False) -> dict:
    """d: a test `Dev` holding the device inputs, output and workspace of a finished run.
    mxfp8: the run was moe_mxfp4w_mxfp8a_forward (MXFP8 activations, reading R18)."""
    inp = d.inp
    T, H, I, E, K = inp.T, inp.H, inp.I, inp.E, inp.K
    routed = inp.topk_ids is not None
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    cdiv = 1 if mxfp8 else 2                                   # activation elements per code byte
    quant = oracle.act_quant_mxfp8 if mxfp8 else oracle.act_quant_mxfp4
    values = oracle.mxfp8_values if mxfp8 else oracle.mxfp4_values
    decisions = check_mx8_requant_decisions if mxfp8 else check_requant_decisions
    L = (mx.moe_mxfp4w_mxfp8a_workspace_layout if mxfp8 else mx.moe_mxfp4_workspace_layout)(T, H, I, E, K, routed)
    R = T * K if routed else T
    out_gpu = bf16_host(d.out)[tok]
    ids = inp.topk_ids[tok].astype(np.int64) if routed else np.zeros((tok.size, 1), np.int64)
    if routed:
        row_of = _ws_view(d.ws, L["row_of"], T, K, "i32")[tok]
    else:
        row_of = tok[:, None]

    # 1. first quantisation, bit-exact
    xq_ref, xs_ref = quant(inp.x[tok])
    xq_all = _ws_view(d.ws, L["xq"], R, H // cdiv)
    hq_all = _ws_view(d.ws, L["hq"], R, I // cdiv)
    if mxfp8 or not routed:
        xs_all = _ws_view(d.ws, L["xs"], R, H // 32)
        hs_all = _ws_view(d.ws, L["hs"], R, I // 32)
    else:   # the routed MXFP4 forward keeps them stage-major
        xs_all = _ws_scales_stage_major(d.ws, L, L["xs"], R, H, routed, E, T)
        hs_all = _ws_scales_stage_major(d.ws, L, L["hs"], R, I, routed, E, T)
    y_all = _ws_view(d.ws, L["y"], R, H, "bf16") if routed else None
    for j in range(ids.shape[1]):
        live = (ids[:, j] >= 0) & (ids[:, j] < E)
        rows = row_of[live, j]
        np.testing.assert_array_equal(xq_all[rows], xq_ref[live], err_msg="xq")
        np.testing.assert_array_equal(xs_all[rows], xs_ref[live], err_msg="xs")
    xv = values(xq_ref, xs_ref)

    flips = _Flips(tok.size, ids.shape[1], FLIP_FRAC_E4M3 if mxfp8 else FLIP_FRAC)
    y_cond = np.zeros((tok.size, ids.shape[1], H))
    for e in range(E):
        sel = np.argwhere((ids == e))
        if sel.size == 0:
            continue
        i_s, k_s = sel[:, 0], sel[:, 1]
        rows = row_of[i_s, k_s]
        W13 = oracle.mxfp4_values(inp.w13[e], inp.s13[e])
        gu = xv[i_s] @ W13.T
        agu = np.abs(xv[i_s]) @ np.abs(W13).T
        del W13
        flips.add(i_s, k_s, *decisions(gu[:, :I], gu[:, I:], agu[:, :I], agu[:, I:], hq_all[rows], hs_all[rows]))
        # 3. L2 on the GPU's own decisions
        W2 = oracle.mxfp4_values(inp.w2[e], inp.s2[e])
        hv = values(hq_all[rows], hs_all[rows])
        exact = hv @ W2.T
        if routed:
            assert_gemm_close(y_all[rows], exact, np.abs(hv) @ np.abs(W2).T, f"L2 expert {e}")
        y_cond[i_s, k_s] = oracle.bf16_bits_to_f64(oracle.bf16_bits_from_f64(exact))
    # 4. output against the oracle on the same decisions
    if routed:
        ref_cond = oracle.moe_combine(y_cond, ids, inp.topk_w[tok], E)
        stats = assert_moe_close(out_gpu, ref_cond, "out vs oracle on the GPU's re-quant decisions")
    else:
        stats = assert_moe_close(out_gpu, oracle.bf16_bits_from_f64(y_cond[:, 0]),
                                 "out vs oracle on the GPU's re-quant decisions")
    forward = oracle.moe_mxfp8_forward if mxfp8 else oracle.moe_forward
    ref = forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.w2, inp.s2, I, tokens=tok)
    return _unconditioned(stats, flips, out_gpu, ref)


class _Flips:
    """Step 2's tally: blocks checked, blocks whose decision differs from the oracle's, blocks
    at risk, and which (token, slot) rows hold a differing block."""

    def __init__(self, n, K, frac=FLIP_FRAC):
        self.blocks = self.differ = self.at_risk = 0
        self.frac = frac
        self.row = np.zeros((n, K), dtype=bool)

    def add(self, i_s, k_s, differ, at_risk):
        self.blocks += differ.size
        self.differ += int(differ.sum())
        self.at_risk += at_risk
        self.row[i_s, k_s] |= differ.any(-1)

    def check(self):
        cap = flip_cap(self.blocks, self.frac)
        assert self.differ <= cap, (f"{self.differ} of {self.blocks} re-quant blocks differ from the oracle's "
                                    f"decision (cap {cap}; {self.at_risk} at risk)")
        return cap


def _unconditioned(stats, flips, out_gpu, ref):
    """Step 4 against the plain oracle: cosine over the sample, the per-element bound on
    every token whose re-quant decisions all equal the oracle's."""
    cap = flips.check()
    g, r = bits_to_f64(out_gpu), bits_to_f64(ref)
    cos = cosine(g, r)
    assert cos >= MOE_COS, f"cosine vs the unconditioned oracle {cos:.6f} < {MOE_COS}"
    err = np.abs(g - r)
    bound = MOE_REL * np.abs(r).max() + MOE_ABS
    clean = ~flips.row.any(-1)
    err_clean = float(err[clean].max()) if clean.any() else 0.0
    assert err_clean <= bound, (f"unconditioned max |err| {err_clean:.4g} > {bound:.4g} on tokens whose re-quant "
                                f"decisions all equal the oracle's")
    stats.update(requant_blocks=flips.blocks, requant_blocks_differing=flips.differ,
                 requant_blocks_at_risk=flips.at_risk, requant_flip_cap=cap, e2e_cos=cos,
                 e2e_max_err=float(err.max()), e2e_max_err_clean_tokens=err_clean, e2e_bound=float(bound),
                 clean_tokens=int(clean.sum()), tokens=int(clean.size))
    return stats


# ----------------------------------------------------------------------------- NVFP4 forward

def _nv_scale_bytes(amax, global_scale):
    """The E4M3 scale byte the NVFP4 quantiser picks for a block maximum (its float32 steps)."""
    f32 = np.float32
    r = f32(1.0) / (f32(6.0) * f32(global_scale))
    with np.errstate(over="ignore"):
        t = np.minimum(np.asarray(amax).astype(np.float32) * r, f32(448.0))
    return oracle.e4m3_round_code(t.astype(np.float64)).astype(np.int64)


def check_nv_requant_decisions(g, u, absg, absu, hq_gpu, hs_gpu, h_global):
    """Step 2 for NVFP4: every GPU block (E4M3 scale + 16 codes) must be the NVFP4
    quantisation of some h' in the interval the float32 accumulation and SiLU allow around
    the oracle's h. g, u, absg, absu already carry the global scales. Returns (differ
    [n, I/16], at_risk) as check_requant_decisions."""
    n, I = g.shape
    to = oracle.bf16_bits_to_f64
    fr = oracle.bf16_bits_from_f64
    eg, eu = absg * ACC_ALLOW, absu * ACC_ALLOW
    gs = [to(fr(g - eg)), to(fr(g + eg))]
    us = [to(fr(u - eu)), to(fr(u + eu))]
    with np.errstate(over="ignore"):
        corners = np.stack([gg / (1.0 + np.exp(-gg)) * uu for gg in gs for uu in us])
    lo = corners.min(0)
    hi = corners.max(0)
    lo = lo - np.abs(lo) * SILU_ALLOW
    hi = hi + np.abs(hi) * SILU_ALLOW
    h_lo, h_hi = to(fr(lo)), to(fr(hi))
    mag_lo = np.where((h_lo <= 0) & (h_hi >= 0), 0.0, np.minimum(np.abs(h_lo), np.abs(h_hi)))
    mag_hi = np.maximum(np.abs(h_lo), np.abs(h_hi))
    nb = I // 16
    S_lo = _nv_scale_bytes(mag_lo.reshape(n, nb, 16).max(-1), h_global)
    S_hi = _nv_scale_bytes(mag_hi.reshape(n, nb, 16).max(-1), h_global)
    hs = hs_gpu.astype(np.int64)
    bad_scale = (hs < S_lo) | (hs > S_hi) | (hs >= 0x7F)
    assert not bad_scale.any(), (f"NVFP4 re-quant scale outside the admissible range at "
                                 f"{np.argwhere(bad_scale)[0].tolist()}")
    f32 = np.float32
    d = oracle.e4m3fn_decode(hs).astype(np.float32) * f32(h_global)
    with np.errstate(divide="ignore"):
        rd = np.repeat(f32(1.0) / d, 16, axis=1)
    zero = np.repeat(hs == 0, 16, axis=1)
    nib = oracle.unpack_nibbles(hq_gpu)
    v_gpu = _signed_code_value(nib & 7, (nib >> 3).astype(bool))

    def qv(h):
        with np.errstate(over="ignore", invalid="ignore"):
            s = h.astype(np.float32) * np.where(zero, f32(0.0), rd)
        s = s.astype(np.float64)
        return _signed_code_value(_e2m1_round_magnitude(np.minimum(np.abs(s), 6.0)), np.signbit(s))

    v_lo, v_hi = qv(h_lo), qv(h_hi)
    bad = (v_gpu < np.minimum(v_lo, v_hi)) | (v_gpu > np.maximum(v_lo, v_hi)) | (zero & (v_gpu != 0))
    assert not bad.any(), (f"NVFP4 re-quant code outside the admissible range at {np.argwhere(bad)[0].tolist()}: "
                           f"gpu {v_gpu[bad][0]}, admissible [{v_lo[bad][0]}, {v_hi[bad][0]}]")
    ref_q, ref_s = oracle.nvfp4_quantize(oracle.swiglu_bf16(g, u), h_global)
    differ = (ref_s != hs_gpu) | (oracle.unpack_nibbles(ref_q).reshape(n, nb, 16) !=
                                  nib.reshape(n, nb, 16)).any(-1)
    at_risk = (S_lo != S_hi) | (v_lo != v_hi).reshape(n, nb, 16).any(-1)
    return differ, int(at_risk.sum())


def check_nvfp4_moe_run(mx, d, tokens=None) -> dict:
    """check_moe_run for a finished moe_nvfp4_forward (d holds an NvMoEInputs)."""
    inp = d.inp
    T, H, I, E, K = inp.T, inp.H, inp.I, inp.E, inp.K
    routed = inp.topk_ids is not None
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    L = mx.moe_nvfp4_workspace_layout(T, H, I, E, K, routed)
    R = T * K if routed else T
    out_gpu = bf16_host(d.out)[tok]
    ids = inp.topk_ids[tok].astype(np.int64) if routed else np.zeros((tok.size, 1), np.int64)
    row_of = _ws_view(d.ws, L["row_of"], T, K, "i32")[tok] if routed else tok[:, None]
    gx, gh = float(np.float32(inp.x_global)), float(np.float32(inp.h_global))

    # 1. first quantisation, bit-exact
    xq_ref, xs_ref = oracle.nvfp4_quantize(inp.x[tok], inp.x_global)
    xq_all = _ws_view(d.ws, L["xq"], R, H // 2)
    hq_all = _ws_view(d.ws, L["hq"], R, I // 2)
    if routed:   # the routed NVFP4 forward keeps them stage-major
        xs_all = _ws_scales_stage_major(d.ws, L, L["xs"], R, H, routed, E, T, block=16)
        hs_all = _ws_scales_stage_major(d.ws, L, L["hs"], R, I, routed, E, T, block=16)
    else:
        xs_all = _ws_view(d.ws, L["xs"], R, H // 16)
        hs_all = _ws_view(d.ws, L["hs"], R, I // 16)
    y_all = _ws_view(d.ws, L["y"], R, H, "bf16") if routed else None
    for j in range(ids.shape[1]):
        live = (ids[:, j] >= 0) & (ids[:, j] < E)
        rows = row_of[live, j]
        np.testing.assert_array_equal(xq_all[rows], xq_ref[live], err_msg="xq")
        np.testing.assert_array_equal(xs_all[rows], xs_ref[live], err_msg="xs")
    xv = oracle.nvfp4_values(xq_ref, xs_ref, 1.0)

    flips = _Flips(tok.size, ids.shape[1])
    y_cond = np.zeros((tok.size, ids.shape[1], H))
    for e in range(E):
        sel = np.argwhere(ids == e)
        if sel.size == 0:
            continue
        i_s, k_s = sel[:, 0], sel[:, 1]
        rows = row_of[i_s, k_s]
        W13 = oracle.nvfp4_values(inp.w13[e], inp.s13[e], 1.0)
        gu = xv[i_s] @ W13.T
        agu = np.abs(xv[i_s]) @ np.abs(W13).T
        del W13
        ag, au = gx * float(inp.g13[e, 0]), gx * float(inp.g13[e, 1])
        flips.add(i_s, k_s, *check_nv_requant_decisions(gu[:, :I] * ag, gu[:, I:] * au, agu[:, :I] * abs(ag),
                                                         agu[:, I:] * abs(au), hq_all[rows], hs_all[rows], gh))
        # 3. L2 on the GPU's own decisions
        W2 = oracle.nvfp4_values(inp.w2[e], inp.s2[e], 1.0)
        hv = oracle.nvfp4_values(hq_all[rows], hs_all[rows], 1.0)
        a2 = gh * float(inp.g2[e])
        exact = (hv @ W2.T) * a2
        if routed:
            assert_gemm_close(y_all[rows], exact, (np.abs(hv) @ np.abs(W2).T) * abs(a2), f"L2 expert {e}")
        y_cond[i_s, k_s] = oracle.bf16_bits_to_f64(oracle.bf16_bits_from_f64(exact))
    # 4. output against the oracle on the same decisions, and against the plain oracle
    if routed:
        ref_cond = oracle.moe_combine(y_cond, ids, inp.topk_w[tok], E)
    else:
        ref_cond = oracle.bf16_bits_from_f64(y_cond[:, 0])
    stats = assert_moe_close(out_gpu, ref_cond, "out vs oracle on the GPU's re-quant decisions")
    ref = oracle.moe_nvfp4_forward(inp.x, inp.topk_ids, inp.topk_w, inp.w13, inp.s13, inp.g13, inp.w2, inp.s2,
                                   inp.g2, inp.x_global, inp.h_global, I, tokens=tok)
    return _unconditioned(stats, flips, out_gpu, ref)
