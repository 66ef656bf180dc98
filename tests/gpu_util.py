"""Helpers for the GPU parity tests: building the library once, moving numpy inputs to the
device, and the comparison rules (bit-exact for codes/scales/dequant; the MoE tolerance
|err| <= 2e-2 * max|ref| + 1e-3 per element with cosine >= 0.9999)."""
from __future__ import annotations

import numpy as np

MOE_REL = 2e-2
MOE_ABS = 1e-3
MOE_COS = 0.9999

_built = False

# Canary guard bands (the stand-in for an out-of-bounds checker, which this pool does not
# offer): a guarded tensor sits inside a larger device buffer whose bytes before and after
# it hold CANARY; check_canaries() asserts that no kernel wrote into them.
CANARY = 0xA5
GUARD_BYTES = 4096                 # a multiple of 256: the tensor keeps the workspace alignment
_guarded: list = []


def native():
    """Build (once per process) and return the binding module."""
    global _built
    import fp4_block_scaled_mxfp4_gb300 as m
    if not _built:
        from fp4_block_scaled_mxfp4_gb300 import build
        build.build()
        _built = True
    return m


def guarded_empty(shape, dtype, guard: int = GUARD_BYTES):
    """An uninitialised device tensor with canary-filled guard bands on both sides."""
    import torch
    shape = tuple(int(v) for v in (shape if isinstance(shape, (tuple, list)) else (shape,)))
    nbytes = int(np.prod(shape, dtype=np.int64)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((guard + nbytes + guard,), CANARY, dtype=torch.uint8, device="cuda")
    t = raw[guard: guard + nbytes].view(dtype).view(shape)
    _guarded.append((raw, guard, nbytes))
    return t


def check_canaries() -> int:
    """Assert every guard band registered since the last call is intact; returns how many
    buffers were checked."""
    bufs = list(_guarded)
    _guarded.clear()
    for raw, guard, nbytes in bufs:
        before = raw[:guard].cpu().numpy()            # only the bands come back to the host
        after = raw[guard + nbytes:].cpu().numpy()
        for name, band in (("before", before), ("after", after)):
            bad = np.nonzero(band != CANARY)[0]
            assert bad.size == 0, (f"a kernel wrote {bad.size} byte(s) into the guard band {name} a buffer of "
                                   f"{nbytes} bytes (first at offset {int(bad[0])} of the band)")
    return len(bufs)


def dev(a: np.ndarray, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_host(t) -> np.ndarray:
    """Device tensor of BF16 (or uint16 bits) -> numpy uint16 bits."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = a.ravel().astype(np.float64)
    b = b.ravel().astype(np.float64)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def assert_moe_close(got_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> dict:
    got = bits_to_f64(got_bits)
    ref = bits_to_f64(ref_bits)
    assert np.isfinite(got).all(), f"{what}: non-finite values in the GPU output"
    assert np.isfinite(ref).all(), f"{what}: non-finite values in the oracle output"
    err = np.abs(got - ref)
    bound = MOE_REL * np.abs(ref).max() + MOE_ABS
    cos = cosine(got, ref)
    stats = dict(max_err=float(err.max()), bound=float(bound), cos=cos,
                 exact_frac=float((got_bits == ref_bits).mean()))
    assert err.max() <= bound, f"{what}: max |err| {err.max():.4g} > {bound:.4g} ({stats})"
    assert cos >= MOE_COS, f"{what}: cosine {cos:.6f} < {MOE_COS} ({stats})"
    return stats


def assert_gemm_close(got_bits: np.ndarray, exact: np.ndarray, absdot: np.ndarray, what: str = ""):
    """GPU BF16(fp32 accumulation) vs the exact product: within one BF16 rounding of the
    exact value plus the float32 accumulation error bound K * 2^-24 * sum|a||b|."""
    got = bits_to_f64(got_bits)
    K_bound = absdot * 2.0 ** -14                     # generous fp32 accumulation allowance
    ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(exact), 1e-300))[1] - 8)
    tol = ulp + K_bound
    err = np.abs(got - exact)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements off; first at "
                           f"{np.argwhere(bad)[0].tolist()} got {got[bad][0]} want {exact[bad][0]}")
