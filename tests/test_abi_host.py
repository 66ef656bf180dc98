"""Host-side checks of the C-ABI library (no GPU needed).

The library must build, load, and export every function include/mxfp4moe.h declares.
Argument validation happens before any CUDA call, so the documented status codes for
bad sizes, null pointers, misaligned pointers and short workspaces are checked here with
fake (never dereferenced) addresses.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4moe.h")

MX_OK, MX_ERR_INVALID_ARG, MX_ERR_UNSUPPORTED, MX_ERR_MISALIGNED, MX_ERR_WORKSPACE = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def lib():
    from fp4_block_scaled_mxfp4_gb300 import build
    build.build()
    from fp4_block_scaled_mxfp4_gb300 import _native
    return _native.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("mxfp4_dequant", "fp8_block_dequant_128x128", "act_quant_mxfp4", "moe_mxfp4_forward",
                 "moe_mxfp4_workspace_size", "mx_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_check_workspace_validation(lib):
    assert lib.mx_check_workspace(None, 1, None) == MX_ERR_INVALID_ARG
    assert lib.mx_check_workspace(FAKE + 16, 1, None) == MX_ERR_MISALIGNED
    assert lib.mx_selftest_wait_timeout_ws(None, None) == MX_ERR_INVALID_ARG
    assert lib.mx_selftest_wait_timeout_ws(FAKE + 16, None) == MX_ERR_MISALIGNED


def test_mxfp8_path_validation(lib):
    assert lib.act_quant_mxfp8(FAKE, FAKE, FAKE, 4, 48, None) == MX_ERR_UNSUPPORTED              # K % 32
    assert lib.act_quant_mxfp8(ODD, FAKE, FAKE, 4, 64, None) == MX_ERR_MISALIGNED
    assert lib.act_quant_mxfp8(FAKE, FAKE, FAKE, 0, 64, None) == MX_OK                           # nothing to do
    assert lib.mxfp8_mxfp4_gemm_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 256, 192, None) == MX_ERR_UNSUPPORTED
    assert lib.mxfp8_mxfp4_gemm_bf16(FAKE, FAKE, FAKE + 16, FAKE, FAKE, 8, 256, 256, None) == MX_ERR_MISALIGNED
    assert lib.mxfp8_mxfp4_gemm_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 256, 256, None) == MX_OK
    # the forward: B operands must be 32-byte aligned; workspace sized for one code byte per element
    T, H, I, E, K = 8, 256, 256, 4, 2
    n8 = lib.moe_mxfp4w_mxfp8a_workspace_size(T, H, I, E, K, 1)
    assert n8 > 0 and lib.moe_mxfp4_workspace_size(T, H, I, E, K, 1) > 0
    # where the codes dominate (the MXFP4 forward rounds its scales up to whole 128-row tiles)
    big = (8192, 7168, 3072, 48, 8, 1)
    assert lib.moe_mxfp4w_mxfp8a_workspace_size(*big) > lib.moe_mxfp4_workspace_size(*big)
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, T, H, I, E, K]
    assert lib.moe_mxfp4w_mxfp8a_forward(*args, FAKE, n8 - 1, None) == MX_ERR_WORKSPACE
    bad = list(args)
    bad[3] = FAKE + 16                                                                        # w13
    assert lib.moe_mxfp4w_mxfp8a_forward(*bad, FAKE, n8, None) == MX_ERR_MISALIGNED
    assert lib.moe_mxfp4w_mxfp8a_forward(FAKE, FAKE, None, *args[3:], FAKE, n8, None) == MX_ERR_INVALID_ARG


def test_status_strings(lib):
    assert lib.mx_status_string(0) == b"MX_OK"
    assert lib.mx_status_string(4) == b"MX_ERR_WORKSPACE"
    assert lib.mx_status_string(99) == b"MX_ERR_UNKNOWN"
    assert lib.mx_version() >= 100


FAKE = 1 << 20          # 16- and 256-byte aligned, never dereferenced
ODD = FAKE + 8          # not 16-byte aligned


def test_dequant_validation(lib):
    assert lib.mxfp4_dequant(FAKE, FAKE, FAKE, 4, 48, None) == MX_ERR_UNSUPPORTED     # cols % 32
    assert lib.mxfp4_dequant(FAKE, FAKE, FAKE, -1, 64, None) == MX_ERR_INVALID_ARG
    assert lib.mxfp4_dequant(FAKE, FAKE, FAKE, 0, 64, None) == MX_OK                  # nothing to do
    assert lib.mxfp4_dequant(None, FAKE, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.mxfp4_dequant(ODD, FAKE, FAKE, 4, 64, None) == MX_ERR_MISALIGNED
    assert lib.fp8_block_dequant_128x128(FAKE, FAKE, FAKE, 4, 40, None) == MX_ERR_UNSUPPORTED
    assert lib.fp8_block_dequant_128x128(FAKE, FAKE, ODD, 4, 64, None) == MX_ERR_MISALIGNED
    assert lib.nvfp4_dequant(FAKE, FAKE, 1.0, FAKE, 4, 40, None) == MX_ERR_UNSUPPORTED     # cols % 16
    assert lib.nvfp4_dequant(FAKE, FAKE, 1.0, FAKE, -1, 64, None) == MX_ERR_INVALID_ARG
    assert lib.nvfp4_dequant(FAKE, FAKE, 1.0, FAKE, 0, 64, None) == MX_OK
    assert lib.nvfp4_dequant(FAKE, None, 1.0, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.nvfp4_dequant(FAKE + 4, FAKE, 1.0, FAKE, 4, 64, None) == MX_ERR_MISALIGNED  # codes 8-byte
    assert lib.nvfp4_dequant(FAKE, FAKE, 1.0, ODD, 4, 64, None) == MX_ERR_MISALIGNED        # out 16-byte
    assert lib.act_quant_mxfp4(FAKE, FAKE, FAKE, 4, 40, None) == MX_ERR_UNSUPPORTED
    assert lib.act_quant_mxfp4(FAKE, None, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG


def test_tiled_scales_validation(lib):
    assert lib.mxfp4_tiled_scales_bytes(300, 7168) == 3 * 56 * 512
    assert lib.mxfp4_tiled_scales_bytes(300, 7200) == 0
    assert lib.mxfp4_scales_to_tiled(FAKE, FAKE, 4, 96, None) == MX_ERR_UNSUPPORTED
    assert lib.mxfp4_scales_to_tiled(FAKE, None, 4, 128, None) == MX_ERR_INVALID_ARG
    assert lib.mxfp4_scales_to_tiled(ODD, FAKE, 4, 128, None) == MX_ERR_MISALIGNED
    assert lib.mxfp4_scales_to_tiled(FAKE, FAKE, 0, 128, None) == MX_OK


def test_gemm_validation(lib):
    assert lib.mxfp4_gemm_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 192, None) == MX_ERR_UNSUPPORTED  # K % 128
    assert lib.mxfp4_gemm_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 250, 256, None) == MX_ERR_UNSUPPORTED
    assert lib.mxfp4_gemm_bf16(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 256, 256, None) == MX_OK
    assert lib.mxfp4_gemm_bf16(FAKE, FAKE, None, FAKE, FAKE, 4, 256, 256, None) == MX_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_bf16(FAKE, ODD, FAKE, FAKE, FAKE, 4, 256, 256, None) == MX_ERR_MISALIGNED
    # NVFP4: every call below is rejected (or has M == 0) before anything launches
    assert lib.nvfp4_gemm_bf16(FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, 4, 256, 192, None) == MX_ERR_UNSUPPORTED  # K % 128
    assert lib.nvfp4_gemm_bf16(FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, 4, 250, 256, None) == MX_ERR_UNSUPPORTED
    assert lib.nvfp4_gemm_bf16(FAKE, FAKE, 1.0, FAKE, FAKE, 1.0, FAKE, 0, 256, 256, None) == MX_OK
    assert lib.nvfp4_gemm_bf16(FAKE, FAKE, 1.0, None, FAKE, 1.0, FAKE, 4, 256, 256, None) == MX_ERR_INVALID_ARG
    assert lib.nvfp4_gemm_bf16(FAKE, FAKE, 1.0, FAKE, ODD, 1.0, FAKE, 4, 256, 256, None) == MX_ERR_MISALIGNED
    assert lib.nvfp4_tiled_scales_bytes(300, 7168) == 3 * 112 * 512
    assert lib.nvfp4_tiled_scales_bytes(300, 7200) == 0
    assert lib.nvfp4_scales_to_tiled(FAKE, FAKE, 4, 96, None) == MX_ERR_UNSUPPORTED
    assert lib.nvfp4_scales_to_tiled(ODD, FAKE, 4, 128, None) == MX_ERR_MISALIGNED
    assert lib.nvfp4_scales_to_tiled(FAKE, FAKE, 0, 128, None) == MX_OK


def _fwd(lib, ids=FAKE, w=FAKE, T=16, H=256, I=128, E=4, K=2, ws=FAKE, ws_bytes=None, x=FAKE):
    if ws_bytes is None:
        ws_bytes = lib.moe_mxfp4_workspace_size(T, H, I, E, K, 1 if ids else 0)
    return lib.moe_mxfp4_forward(x, ids, w, FAKE, FAKE, FAKE, FAKE, FAKE, T, H, I, E, K, ws, ws_bytes, None)


def test_forward_validation(lib):
    assert _fwd(lib, H=200) == MX_ERR_UNSUPPORTED
    assert _fwd(lib, I=96) == MX_ERR_UNSUPPORTED
    assert _fwd(lib, E=0) == MX_ERR_INVALID_ARG
    assert _fwd(lib, E=2000) == MX_ERR_UNSUPPORTED
    assert _fwd(lib, K=0) == MX_ERR_INVALID_ARG
    assert _fwd(lib, K=65) == MX_ERR_UNSUPPORTED
    assert _fwd(lib, T=-1) == MX_ERR_INVALID_ARG
    assert _fwd(lib, T=0) == MX_OK
    assert _fwd(lib, w=None) == MX_ERR_INVALID_ARG                  # ids without weights
    assert _fwd(lib, ids=None, w=None, E=2) == MX_ERR_INVALID_ARG  # shared mode needs E = 1
    assert _fwd(lib, x=None) == MX_ERR_INVALID_ARG
    assert _fwd(lib, x=ODD) == MX_ERR_MISALIGNED
    need = lib.moe_mxfp4_workspace_size(16, 256, 128, 4, 2, 1)
    assert need > 0
    assert _fwd(lib, ws_bytes=need - 1) == MX_ERR_WORKSPACE
    assert _fwd(lib, ws=None) == MX_ERR_WORKSPACE
    assert _fwd(lib, ws=FAKE + 128) == MX_ERR_MISALIGNED
    assert lib.moe_mxfp4_workspace_size(16, 200, 128, 4, 2, 1) == 0   # unsupported sizes -> 0


def test_workspace_size_grows_with_tokens(lib):
    a = lib.moe_mxfp4_workspace_size(64, 7168, 3072, 48, 8, 1)
    b = lib.moe_mxfp4_workspace_size(8192, 7168, 3072, 48, 8, 1)
    s = lib.moe_mxfp4_workspace_size(256, 7168, 3072, 1, 1, 0)
    assert 0 < a < b and s > 0
    assert a % 256 == 0 and b % 256 == 0
    # the routed workspace holds at least the quantised activations and the L2 output
    assert b >= 8192 * 8 * (7168 // 2 + 7168 * 2)


def test_route_validation(lib):
    need = lib.moe_mxfp4_workspace_size(10, 128, 128, 4, 2, 1)
    assert lib.moe_mxfp4_route(FAKE, 10, 2, 4, FAKE, FAKE, FAKE, FAKE, need - 1, None) == MX_ERR_WORKSPACE
    assert lib.moe_mxfp4_route(FAKE, 10, 2, 0, FAKE, FAKE, FAKE, FAKE, need, None) == MX_ERR_INVALID_ARG
    assert lib.moe_mxfp4_route(None, 10, 2, 4, FAKE, FAKE, FAKE, FAKE, need, None) == MX_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from fp4_block_scaled_mxfp4_gb300 import _native
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _native.lib()


def test_nvfp4_quant_and_forward_validation(lib):
    """Every call is rejected (or has nothing to do) before anything launches."""
    assert lib.act_quant_nvfp4(FAKE, 1.0, FAKE, FAKE, 4, 40, None) == MX_ERR_UNSUPPORTED       # K % 16
    assert lib.act_quant_nvfp4(FAKE, 0.0, FAKE, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG       # global 0
    assert lib.act_quant_nvfp4(FAKE, float("nan"), FAKE, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.act_quant_nvfp4(FAKE, 2.0 ** -120, FAKE, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.act_quant_nvfp4(FAKE, 2.0 ** 101, FAKE, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.act_quant_nvfp4(FAKE, 1.0, None, FAKE, 4, 64, None) == MX_ERR_INVALID_ARG
    assert lib.act_quant_nvfp4(FAKE, 1.0, FAKE + 4, FAKE, 4, 64, None) == MX_ERR_MISALIGNED   # codes 8-byte
    assert lib.act_quant_nvfp4(FAKE, 1.0, FAKE, FAKE, 0, 64, None) == MX_OK

    def fwd(ids=FAKE, w=FAKE, g13=FAKE, g2=FAKE, gx=0.01, gh=0.25, T=16, H=256, I=128, E=4, K=2, ws=FAKE,
            ws_bytes=None):
        if ws_bytes is None:
            ws_bytes = lib.moe_nvfp4_workspace_size(T, H, I, E, K, 1 if ids else 0)
        return lib.moe_nvfp4_forward(FAKE, ids, w, FAKE, FAKE, g13, FAKE, FAKE, g2, gx, gh, FAKE, T, H, I, E, K,
                                     ws, ws_bytes, None)

    assert fwd(H=200) == MX_ERR_UNSUPPORTED
    assert fwd(gx=0.0) == MX_ERR_INVALID_ARG
    assert fwd(gh=float("inf")) == MX_ERR_INVALID_ARG
    assert fwd(g13=None) == MX_ERR_INVALID_ARG
    assert fwd(g2=None) == MX_ERR_INVALID_ARG
    assert fwd(w=None) == MX_ERR_INVALID_ARG
    assert fwd(ids=None, w=None, E=2) == MX_ERR_INVALID_ARG
    assert fwd(T=0) == MX_OK
    need = lib.moe_nvfp4_workspace_size(16, 256, 128, 4, 2, 1)
    n4 = lib.moe_mxfp4_workspace_size(16, 256, 128, 4, 2, 1)
    assert n4 < need < 2 * n4             # the MXFP4 layout with twice the scale bytes
    assert fwd(ws_bytes=need - 1) == MX_ERR_WORKSPACE
    assert fwd(ws=FAKE + 128) == MX_ERR_MISALIGNED
    # the scale regions hold one byte per 16 columns
    buf = (ctypes.c_int64 * 8)()
    assert lib.moe_nvfp4_workspace_layout(16, 256, 128, 4, 2, 1, ctypes.addressof(buf)) == MX_OK
    xs, hq = buf[1], buf[2]
    assert hq - xs >= 32 * (256 // 16)


def test_nvfp4_fused_projection_validation(lib):
    """Every call is rejected (or has M == 0) before anything launches."""
    def call(rows, globals_=None, M=4, K=256, b=FAKE):
        n = len(rows)
        gl = (ctypes.c_float * max(n, 1))(*([0.5] * n if globals_ is None else globals_))
        rr = (ctypes.c_int64 * max(n, 1))(*rows)
        return lib.nvfp4_gemm_bf16_multi(FAKE, FAKE, 1.0, b, FAKE, ctypes.addressof(gl), ctypes.addressof(rr), n,
                                         FAKE, M, K, None)
    assert call([1536, 520]) == MX_ERR_UNSUPPORTED                 # a segment not a multiple of 16
    assert call([1536, 0]) == MX_ERR_INVALID_ARG
    assert call([]) == MX_ERR_INVALID_ARG
    assert call([16] * 9) == MX_ERR_UNSUPPORTED                    # more than 8 segments
    assert call([1536, 576], K=192) == MX_ERR_UNSUPPORTED           # K % 128
    assert call([1536, 576], M=0) == MX_OK
    assert call([1536, 576], b=None) == MX_ERR_INVALID_ARG
    assert call([1536, 576], b=ODD) == MX_ERR_MISALIGNED
