"""Thin ctypes binding of the C ABI in include/mxfp4moe.h (argument marshalling only).

Every function takes torch CUDA tensors, checks dtype / shape / contiguity, passes raw
device pointers and sizes to the library, and raises ``MXError`` on a non-zero status.
All arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch fallback:
if ``libmxfp4moe.so`` is missing or cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmxfp4moe.so")
_lib: Optional[ctypes.CDLL] = None

_c_i64 = ctypes.c_int64
_c_ptr = ctypes.c_void_p

# name -> (restype, argtypes)
_SIGNATURES = {
    "mx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mx_version": (ctypes.c_int, []),
    "mx_device_status": (ctypes.c_int, [ctypes.c_int]),
    "mx_selftest_wait_timeout": (ctypes.c_int, [_c_ptr]),
    "mx_selftest_wait_timeout_ws": (ctypes.c_int, [_c_ptr, _c_ptr]),
    "mx_check_workspace": (ctypes.c_int, [_c_ptr, ctypes.c_int, _c_ptr]),
    "mx_selftest_grid_barrier_timeout": (ctypes.c_int, [_c_ptr, _c_ptr]),
    "mxfp4_dequant": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "fp8_block_dequant_128x128": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "nvfp4_dequant": (ctypes.c_int, [_c_ptr, _c_ptr, ctypes.c_float, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "nvfp4_tiled_scales_bytes": (ctypes.c_size_t, [_c_i64, _c_i64]),
    "nvfp4_scales_to_tiled": (ctypes.c_int, [_c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "nvfp4_gemm_bf16": (ctypes.c_int, [_c_ptr, _c_ptr, ctypes.c_float, _c_ptr, _c_ptr, ctypes.c_float, _c_ptr,
                                       _c_i64, _c_i64, _c_i64, _c_ptr]),
    "nvfp4_gemm_bf16_multi": (ctypes.c_int, [_c_ptr, _c_ptr, ctypes.c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                             ctypes.c_int, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "act_quant_mxfp4": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "act_quant_nvfp4": (ctypes.c_int, [_c_ptr, ctypes.c_float, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "act_quant_mxfp8": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "mxfp8_mxfp4_gemm_bf16": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr]),
    "moe_mxfp4w_mxfp8a_workspace_size": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "moe_mxfp4w_mxfp8a_workspace_layout": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int,
                                                           _c_ptr]),
    "moe_mxfp4w_mxfp8a_forward": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                                 _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t,
                                                 _c_ptr]),
    "moe_mxfp4w_mxfp8a_forward_timed": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                                       _c_ptr, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr,
                                                       ctypes.c_size_t, _c_ptr, _c_ptr]),
    "nvfp4_calibrate_global": (ctypes.c_int, [_c_ptr, _c_i64, _c_i64, _c_ptr, _c_ptr, _c_ptr]),
    "moe_nvfp4_workspace_size": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "moe_nvfp4_workspace_layout": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int, _c_ptr]),
    "moe_nvfp4_forward": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                         ctypes.c_float, ctypes.c_float, _c_ptr, _c_i64, _c_i64, _c_i64, _c_i64,
                                         _c_i64, _c_ptr, ctypes.c_size_t, _c_ptr]),
    "moe_nvfp4_forward_timed": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                               _c_ptr, ctypes.c_float, ctypes.c_float, _c_ptr, _c_i64, _c_i64,
                                               _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t, _c_ptr, _c_ptr]),
    "mxfp4_tiled_scales_bytes": (ctypes.c_size_t, [_c_i64, _c_i64]),
    "mxfp4_scales_to_tiled": (ctypes.c_int, [_c_ptr, _c_ptr, _c_i64, _c_i64, _c_ptr]),
    "mxfp4_gemm_bf16": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr]),
    "moe_mxfp4_workspace_size": (ctypes.c_size_t, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int]),
    "moe_mxfp4_forward": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                         _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t,
                                         _c_ptr]),
    "moe_mxfp4_forward_timed": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                               _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t,
                                               _c_ptr, _c_ptr, ctypes.c_int]),
    "moe_mxfp4_forward_tiled": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                               _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t,
                                               _c_ptr]),
    "moe_mxfp4_forward_fused": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                               _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr, ctypes.c_size_t,
                                               _c_ptr]),
    "moe_mxfp4_forward_noalloc": (ctypes.c_int, [_c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                                 _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_ptr]),
    "moe_mxfp4_workspace_layout": (ctypes.c_int, [_c_i64, _c_i64, _c_i64, _c_i64, _c_i64, ctypes.c_int, _c_ptr]),
    "moe_mxfp4_route": (ctypes.c_int, [_c_ptr, _c_i64, _c_i64, _c_i64, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                       ctypes.c_size_t, _c_ptr]),
}

MX_OK = 0


class MXError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libmxfp4moe.so (once). Raises if it is missing: there is no fallback path."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libmxfp4moe.so is not built ({_LIB_PATH}); run "
                               "fp4_block_scaled_mxfp4_gb300.build.build() first")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().mx_status_string(int(status)).decode()


def _check(status: int, call: str) -> None:
    if status != MX_OK:
        raise MXError(status, call)


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _need(t, dtype, shape, name):
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")


def _bf16_like(t):
    import torch
    return t.dtype in (torch.bfloat16, torch.uint16, torch.int16)


def mxfp4_dequant(codes, sf, out, stream=None) -> None:
    """out[r, c] = bf16(E2M1(codes) * 2^(sf - 127)); codes u8 [R, C/2], sf u8 [R, C/32], out [R, C]."""
    import torch
    R, half = codes.shape
    C = 2 * half
    _need(codes, torch.uint8, (R, half), "codes")
    _need(sf, torch.uint8, (R, C // 32), "sf")
    if not _bf16_like(out):
        raise ValueError("out must be bfloat16 (or its 16-bit bit pattern)")
    _need(out, out.dtype, (R, C), "out")
    _check(lib().mxfp4_dequant(_ptr(codes), _ptr(sf), _ptr(out), R, C, _stream(stream)), "mxfp4_dequant")


def nvfp4_dequant(codes, sf, global_scale, out, stream=None) -> None:
    """out[r, c] = bf16(float32(E2M1(codes) * e4m3(sf[r, c/16]) * global_scale));
    codes u8 [R, C/2], sf u8 [R, C/16] (E4M3 bytes), global_scale a float, out [R, C]."""
    import torch
    R, half = codes.shape
    C = 2 * half
    _need(codes, torch.uint8, (R, half), "codes")
    _need(sf, torch.uint8, (R, C // 16), "sf")
    if not _bf16_like(out):
        raise ValueError("out must be bfloat16 (or its 16-bit bit pattern)")
    _need(out, out.dtype, (R, C), "out")
    _check(lib().nvfp4_dequant(_ptr(codes), _ptr(sf), float(global_scale), _ptr(out), R, C, _stream(stream)),
           "nvfp4_dequant")


def nvfp4_tiled_scales_bytes(rows: int, cols: int) -> int:
    return int(lib().nvfp4_tiled_scales_bytes(rows, cols))


def nvfp4_scales_to_tiled(sf, out, stream=None) -> None:
    """NVFP4 scale tensor u8 [rows, cols/16] -> tile layout (u8, nvfp4_tiled_scales_bytes bytes)."""
    import torch
    rows, kb = sf.shape
    _need(sf, torch.uint8, (rows, kb), "sf")
    if out.dtype != torch.uint8 or out.numel() < nvfp4_tiled_scales_bytes(rows, 16 * kb) or not out.is_cuda:
        raise ValueError("out: uint8 CUDA buffer of nvfp4_tiled_scales_bytes bytes")
    _check(lib().nvfp4_scales_to_tiled(_ptr(sf), _ptr(out), rows, 16 * kb, _stream(stream)),
           "nvfp4_scales_to_tiled")


def nvfp4_gemm_bf16(a, sa, a_global, b, sb_tiled, b_global, d, stream=None) -> None:
    """d = bf16(a_global * b_global * A . B^T) for NVFP4 A (a u8 [M, K/2], sa u8 [M, K/16]) and
    B (b u8 [N, K/2], sb_tiled = nvfp4_scales_to_tiled of B's [N, K/16] scales)."""
    import torch
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    _need(a, torch.uint8, (M, half), "a")
    _need(sa, torch.uint8, (M, K // 16), "sa")
    _need(b, torch.uint8, (N, half), "b")
    if sb_tiled.dtype != torch.uint8 or sb_tiled.numel() < nvfp4_tiled_scales_bytes(N, K) or not sb_tiled.is_cuda:
        raise ValueError("sb_tiled: uint8 CUDA buffer of nvfp4_tiled_scales_bytes(N, K) bytes")
    if not _bf16_like(d):
        raise ValueError("d must be bfloat16 (or its 16-bit bit pattern)")
    _need(d, d.dtype, (M, N), "d")
    _check(lib().nvfp4_gemm_bf16(_ptr(a), _ptr(sa), float(a_global), _ptr(b), _ptr(sb_tiled), float(b_global),
                                 _ptr(d), M, N, K, _stream(stream)), "nvfp4_gemm_bf16")


def nvfp4_gemm_bf16_multi(a, sa, a_global, b, sb_tiled, b_globals, seg_rows, d, stream=None) -> None:
    """Fused NVFP4 projection: B stacks len(seg_rows) weight matrices along N (segment s has
    seg_rows[s] rows and global b_globals[s]); d[:, segment s] = bf16(a_global * b_globals[s]
    * A . B_s^T). b_globals / seg_rows are host sequences."""
    import torch
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    if sum(int(r) for r in seg_rows) != N or len(seg_rows) != len(b_globals):
        raise ValueError("seg_rows must cover B's rows, with one global per segment")
    _need(a, torch.uint8, (M, half), "a")
    _need(sa, torch.uint8, (M, K // 16), "sa")
    _need(b, torch.uint8, (N, half), "b")
    if sb_tiled.dtype != torch.uint8 or sb_tiled.numel() < nvfp4_tiled_scales_bytes(N, K) or not sb_tiled.is_cuda:
        raise ValueError("sb_tiled: uint8 CUDA buffer of nvfp4_tiled_scales_bytes(N, K) bytes")
    if not _bf16_like(d):
        raise ValueError("d must be bfloat16 (or its 16-bit bit pattern)")
    _need(d, d.dtype, (M, N), "d")
    n = len(seg_rows)
    gl = (ctypes.c_float * n)(*[float(x) for x in b_globals])
    rows = (ctypes.c_int64 * n)(*[int(x) for x in seg_rows])
    _check(lib().nvfp4_gemm_bf16_multi(_ptr(a), _ptr(sa), float(a_global), _ptr(b), _ptr(sb_tiled),
                                       ctypes.addressof(gl), ctypes.addressof(rows), n, _ptr(d), M, K,
                                       _stream(stream)), "nvfp4_gemm_bf16_multi")


def fp8_block_dequant_128x128(q, sf, out, stream=None) -> None:
    """out = bf16(e4m3(q) * 2^(sf[i/128, j/128] - 127)); q u8 [R, C], sf u8 [ceil(R/128), ceil(C/128)]."""
    import torch
    R, C = q.shape
    _need(q, q.dtype, (R, C), "q")
    if q.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError("q must be uint8 or float8_e4m3fn")
    _need(sf, sf.dtype, ((R + 127) // 128, (C + 127) // 128), "sf")
    _need(out, out.dtype, (R, C), "out")
    _check(lib().fp8_block_dequant_128x128(_ptr(q), _ptr(sf), _ptr(out), R, C, _stream(stream)),
           "fp8_block_dequant_128x128")


def act_quant_mxfp4(x, codes, sf, stream=None) -> None:
    """MX quantisation of BF16 x [M, K] into codes u8 [M, K/2] and E8M0 scales u8 [M, K/32]."""
    import torch
    M, K = x.shape
    _need(x, x.dtype, (M, K), "x")
    _need(codes, torch.uint8, (M, K // 2), "codes")
    _need(sf, torch.uint8, (M, K // 32), "sf")
    _check(lib().act_quant_mxfp4(_ptr(x), _ptr(codes), _ptr(sf), M, K, _stream(stream)), "act_quant_mxfp4")


def act_quant_nvfp4(x, global_scale, codes, sf, stream=None) -> None:
    """NVFP4 quantisation of BF16 x [M, K] against the float32 global: codes u8 [M, K/2],
    E4M3 scales u8 [M, K/16]."""
    import torch
    M, K = x.shape
    _need(x, x.dtype, (M, K), "x")
    _need(codes, torch.uint8, (M, K // 2), "codes")
    _need(sf, torch.uint8, (M, K // 16), "sf")
    _check(lib().act_quant_nvfp4(_ptr(x), float(global_scale), _ptr(codes), _ptr(sf), M, K, _stream(stream)),
           "act_quant_nvfp4")


def nvfp4_calibrate_global(x, amax, global_scale, stream=None) -> None:
    """Warm-up calibration of an NVFP4 activation global on the GPU: folds the largest finite
    |x| of the batch x (bf16 [M, K]) into the running maximum amax (float32 [1], device;
    zero it before the first batch) and writes amax / (6 * 448) to global_scale (float32 [1])."""
    import torch
    M, K = x.shape
    _need(x, x.dtype, (M, K), "x")
    _need(amax, torch.float32, (1,), "amax")
    _need(global_scale, torch.float32, (1,), "global_scale")
    _check(lib().nvfp4_calibrate_global(_ptr(x), M, K, _ptr(amax), _ptr(global_scale), _stream(stream)),
           "nvfp4_calibrate_global")


def act_quant_mxfp8(x, codes, sf, stream=None) -> None:
    """BF16 [M, K] -> MXFP8 codes uint8 [M, K] (E4M3) + E8M0 scales uint8 [M, K/32]."""
    import torch
    M, K = x.shape
    _need(x, x.dtype, (M, K), "x")
    _need(codes, torch.uint8, (M, K), "codes")
    _need(sf, torch.uint8, (M, K // 32), "sf")
    _check(lib().act_quant_mxfp8(_ptr(x), _ptr(codes), _ptr(sf), M, K, _stream(stream)), "act_quant_mxfp8")


def mxfp8_mxfp4_gemm_bf16(a, sa, b, sb_tiled, d, stream=None) -> None:
    """D = bf16(A . B^T): MXFP8 A (codes [M, K], scales [M, K/32]), MXFP4 B (codes [N, K/2],
    tile-layout scales)."""
    import torch
    M, K = a.shape
    N = b.shape[0]
    _need(a, torch.uint8, (M, K), "a")
    _need(sa, torch.uint8, (M, K // 32), "sa")
    _need(b, torch.uint8, (N, K // 2), "b")
    if sb_tiled.dtype != torch.uint8 or sb_tiled.numel() < mxfp4_tiled_scales_bytes(N, K):
        raise ValueError("sb_tiled: expected the tile layout of B's scales")
    _need(d, d.dtype, (M, N), "d")
    _check(lib().mxfp8_mxfp4_gemm_bf16(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb_tiled), _ptr(d), M, N, K,
                                       _stream(stream)), "mxfp8_mxfp4_gemm_bf16")


def moe_mxfp4w_mxfp8a_workspace_size(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> int:
    return int(lib().moe_mxfp4w_mxfp8a_workspace_size(T, H, I, E, K, 1 if routed else 0))


def moe_mxfp4w_mxfp8a_workspace_layout(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> dict:
    """Byte offsets of the intermediates an MXFP8-activation forward leaves in its workspace."""
    buf = (ctypes.c_int64 * 8)()
    _check(lib().moe_mxfp4w_mxfp8a_workspace_layout(T, H, I, E, K, 1 if routed else 0, ctypes.addressof(buf)),
           "moe_mxfp4w_mxfp8a_workspace_layout")
    names = ("xq", "xs", "hq", "hs", "y", "row_of", "counts", "offsets")
    return {n: int(v) for n, v in zip(names, buf)}


def moe_mxfp4w_mxfp8a_forward(x, topk_ids, topk_w, w13, s13_tiled, w2, s2_tiled, out, workspace, stream=None,
                              events=None) -> None:
    """MoE expert FFN with MXFP8 activations over MXFP4 weights (tile-layout weight scales);
    topk_ids/topk_w None selects the shared expert. ``events`` as in moe_mxfp4_forward."""
    import torch
    T, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = topk_ids.shape[1] if topk_ids is not None else 1
    _need(x, x.dtype, (T, H), "x")
    if topk_ids is not None:
        _need(topk_ids, torch.int32, (T, K), "topk_ids")
        _need(topk_w, torch.float32, (T, K), "topk_w")
    _need(w13, torch.uint8, (E, 2 * I, H // 2), "w13")
    _need(w2, torch.uint8, (E, H, I // 2), "w2")
    for t, r, c, n in ((s13_tiled, E * 2 * I, H, "s13_tiled"), (s2_tiled, E * H, I, "s2_tiled")):
        if t.dtype != torch.uint8 or t.numel() < mxfp4_tiled_scales_bytes(r, c) or not t.is_cuda:
            raise ValueError(f"{n}: expected the tile layout of the scales")
    _need(out, out.dtype, (T, H), "out")
    ws_bytes = workspace.numel() * workspace.element_size()
    args = (_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(s13_tiled), _ptr(w2), _ptr(s2_tiled), _ptr(out),
            T, H, I, E, K, _ptr(workspace), ws_bytes, _stream(stream))
    if events is not None:
        evs = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else 0) for e in events])
        _check(lib().moe_mxfp4w_mxfp8a_forward_timed(*args, ctypes.addressof(evs)), "moe_mxfp4w_mxfp8a_forward_timed")
    else:
        _check(lib().moe_mxfp4w_mxfp8a_forward(*args), "moe_mxfp4w_mxfp8a_forward")


def mxfp4_tiled_scales_bytes(rows: int, cols: int) -> int:
    return int(lib().mxfp4_tiled_scales_bytes(rows, cols))


def mxfp4_scales_to_tiled(sf, out, stream=None) -> None:
    """Scale tensor u8 [rows, cols/32] -> tile layout (u8, mxfp4_tiled_scales_bytes bytes)."""
    import torch
    rows, kb = sf.shape
    _need(sf, torch.uint8, (rows, kb), "sf")
    if out.dtype != torch.uint8 or out.numel() < mxfp4_tiled_scales_bytes(rows, 32 * kb) or not out.is_cuda:
        raise ValueError("out: too small for the tile layout")
    _check(lib().mxfp4_scales_to_tiled(_ptr(sf), _ptr(out), rows, 32 * kb, _stream(stream)),
           "mxfp4_scales_to_tiled")


def mxfp4_gemm_bf16(a, sa, b, sb_tiled, d, stream=None) -> None:
    """d = bf16(A . B^T) for MXFP4 A [M, K] (a u8 [M, K/2], sa [M, K/32]) and B [N, K]
    (b u8 [N, K/2], sb_tiled = mxfp4_scales_to_tiled of B's [N, K/32] scales)."""
    import torch
    M, half = a.shape
    N = b.shape[0]
    K = 2 * half
    _need(a, torch.uint8, (M, half), "a")
    _need(sa, torch.uint8, (M, K // 32), "sa")
    _need(b, torch.uint8, (N, half), "b")
    sb = sb_tiled
    if sb.dtype != torch.uint8 or sb.numel() < mxfp4_tiled_scales_bytes(N, K) or not sb.is_cuda:
        raise ValueError("sb_tiled: expected the tile layout of B's scales")
    _need(d, d.dtype, (M, N), "d")
    _check(lib().mxfp4_gemm_bf16(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(d), M, N, K, _stream(stream)),
           "mxfp4_gemm_bf16")


def moe_mxfp4_workspace_size(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> int:
    return int(lib().moe_mxfp4_workspace_size(T, H, I, E, K, 1 if routed else 0))


def moe_mxfp4_workspace_layout(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> dict:
    """Byte offsets of the intermediates a forward leaves in its workspace (see the header)."""
    buf = (ctypes.c_int64 * 8)()
    _check(lib().moe_mxfp4_workspace_layout(T, H, I, E, K, 1 if routed else 0, ctypes.addressof(buf)),
           "moe_mxfp4_workspace_layout")
    names = ("xq", "xs", "hq", "hs", "y", "row_of", "counts", "offsets")
    return {n: int(v) for n, v in zip(names, buf)}


def moe_mxfp4_forward(x, topk_ids, topk_w, w13, s13, w2, s2, out, workspace, stream=None, events=None,
                      scales_tiled=False, fused=False) -> None:
    """MoE expert FFN over MXFP4 weights; topk_ids/topk_w None selects the shared expert.

    s13 / s2: the row-major E8M0 scales ([E, 2I, H/32], [E, H, I/32]), or with
    scales_tiled=True their tile layout (mxfp4_scales_to_tiled; any uint8 buffer of that
    size). ``events``: optional sequence of 6 torch.cuda.Event (or None) recorded at the
    phase boundaries (before, after routing, after quantisation, after L1, after L2, after
    combine). ``fused=True`` (tile-layout scales only) runs the whole forward as one
    persistent kernel launch (moe_mxfp4_forward_fused).
    """
    import torch
    T, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = topk_ids.shape[1] if topk_ids is not None else 1
    _need(x, x.dtype, (T, H), "x")
    if topk_ids is not None:
        _need(topk_ids, torch.int32, (T, K), "topk_ids")
        _need(topk_w, torch.float32, (T, K), "topk_w")
    _need(w13, torch.uint8, (E, 2 * I, H // 2), "w13")
    _need(w2, torch.uint8, (E, H, I // 2), "w2")
    if scales_tiled:
        for t, r, c, n in ((s13, E * 2 * I, H, "s13"), (s2, E * H, I, "s2")):
            if t.dtype != torch.uint8 or t.numel() < mxfp4_tiled_scales_bytes(r, c) or not t.is_cuda:
                raise ValueError(f"{n}: expected the tile layout of the scales")
    else:
        _need(s13, torch.uint8, (E, 2 * I, H // 32), "s13")
        _need(s2, torch.uint8, (E, H, I // 32), "s2")
    _need(out, out.dtype, (T, H), "out")
    ws_bytes = workspace.numel() * workspace.element_size()
    args = (_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), _ptr(out),
            T, H, I, E, K, _ptr(workspace), ws_bytes, _stream(stream))
    if fused:
        if not scales_tiled or events is not None:
            raise ValueError("the single-launch forward takes tile-layout scales and records no phase events")
        _check(lib().moe_mxfp4_forward_fused(*args), "moe_mxfp4_forward_fused")
    elif events is not None:
        evs = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else 0) for e in events])
        _check(lib().moe_mxfp4_forward_timed(*args, ctypes.addressof(evs), 1 if scales_tiled else 0),
               "moe_mxfp4_forward_timed")
    elif scales_tiled:
        _check(lib().moe_mxfp4_forward_tiled(*args), "moe_mxfp4_forward_tiled")
    else:
        _check(lib().moe_mxfp4_forward(*args), "moe_mxfp4_forward")


def moe_nvfp4_workspace_size(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> int:
    return int(lib().moe_nvfp4_workspace_size(T, H, I, E, K, 1 if routed else 0))


def moe_nvfp4_workspace_layout(T: int, H: int, I: int, E: int, K: int, routed: bool = True) -> dict:
    """Byte offsets of the intermediates an NVFP4 forward leaves in its workspace."""
    buf = (ctypes.c_int64 * 8)()
    _check(lib().moe_nvfp4_workspace_layout(T, H, I, E, K, 1 if routed else 0, ctypes.addressof(buf)),
           "moe_nvfp4_workspace_layout")
    names = ("xq", "xs", "hq", "hs", "y", "row_of", "counts", "offsets")
    return {n: int(v) for n, v in zip(names, buf)}


def moe_nvfp4_forward(x, topk_ids, topk_w, w13, s13_tiled, g13, w2, s2_tiled, g2, x_global, h_global, out,
                      workspace, stream=None, events=None) -> None:
    """MoE expert FFN over NVFP4 weights and activations; topk_ids/topk_w None selects the
    shared expert. s13_tiled / s2_tiled: nvfp4_scales_to_tiled of the E4M3 scales
    ([E*2I, H/16], [E*H, I/16]); g13 float32 [E, 2] (gate, up) and g2 float32 [E] on the
    device; x_global / h_global: the activation globals. ``events`` as in moe_mxfp4_forward."""
    import torch
    T, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = topk_ids.shape[1] if topk_ids is not None else 1
    _need(x, x.dtype, (T, H), "x")
    if topk_ids is not None:
        _need(topk_ids, torch.int32, (T, K), "topk_ids")
        _need(topk_w, torch.float32, (T, K), "topk_w")
    _need(w13, torch.uint8, (E, 2 * I, H // 2), "w13")
    _need(w2, torch.uint8, (E, H, I // 2), "w2")
    for t, r, c, n in ((s13_tiled, E * 2 * I, H, "s13_tiled"), (s2_tiled, E * H, I, "s2_tiled")):
        if t.dtype != torch.uint8 or t.numel() < nvfp4_tiled_scales_bytes(r, c) or not t.is_cuda:
            raise ValueError(f"{n}: expected the tile layout of the E4M3 scales")
    _need(g13, torch.float32, (E, 2), "g13")
    _need(g2, torch.float32, (E,), "g2")
    _need(out, out.dtype, (T, H), "out")
    ws_bytes = workspace.numel() * workspace.element_size()
    args = (_ptr(x), _ptr(topk_ids), _ptr(topk_w), _ptr(w13), _ptr(s13_tiled), _ptr(g13), _ptr(w2), _ptr(s2_tiled),
            _ptr(g2), float(x_global), float(h_global), _ptr(out), T, H, I, E, K, _ptr(workspace), ws_bytes,
            _stream(stream))
    if events is not None:
        evs = (ctypes.c_void_p * 6)(*[(e.cuda_event if e is not None else 0) for e in events])
        _check(lib().moe_nvfp4_forward_timed(*args, ctypes.addressof(evs)), "moe_nvfp4_forward_timed")
    else:
        _check(lib().moe_nvfp4_forward(*args), "moe_nvfp4_forward")


def moe_mxfp4_route(topk_ids, E: int, counts, offsets, row_of, workspace, stream=None) -> None:
    """Routing permutation only: counts [E], offsets [E+1], row_of [T, K] (int32)."""
    import torch
    T, K = topk_ids.shape
    _need(topk_ids, torch.int32, (T, K), "topk_ids")
    _need(counts, torch.int32, (E,), "counts")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    _need(row_of, torch.int32, (T, K), "row_of")
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().moe_mxfp4_route(_ptr(topk_ids), T, K, E, _ptr(counts), _ptr(offsets), _ptr(row_of),
                                 _ptr(workspace), ws_bytes, _stream(stream)), "moe_mxfp4_route")


def selftest_wait_timeout(stream=None, workspace=None) -> None:
    """Launch the failure-path self-test: a bounded wait (about 2 s) on a barrier nothing
    arrives at, which records a timeout in the device status word (see device_status) and,
    given a workspace, in that workspace's word (see check_workspace)."""
    if workspace is None:
        _check(lib().mx_selftest_wait_timeout(_stream(stream)), "mx_selftest_wait_timeout")
    else:
        _check(lib().mx_selftest_wait_timeout_ws(_ptr(workspace), _stream(stream)), "mx_selftest_wait_timeout_ws")


def selftest_grid_barrier_timeout(workspace, stream=None) -> None:
    """Launch the grid-barrier failure-path self-test on `workspace` (see the header)."""
    _check(lib().mx_selftest_grid_barrier_timeout(_ptr(workspace), _stream(stream)),
           "mx_selftest_grid_barrier_timeout")


def check_workspace(workspace, stream=None, clear: bool = True) -> int:
    """Wait for `stream` only and return the status of the last forward launched on it with
    this workspace (0 = MX_OK, 6 = MX_ERR_DEVICE_TIMEOUT)."""
    st = int(lib().mx_check_workspace(_ptr(workspace), 1 if clear else 0, _stream(stream)))
    if st not in (MX_OK, 6):
        raise MXError(st, "mx_check_workspace")
    return st


def device_status(clear: bool = True) -> int:
    """Synchronise and return the device status word as a status code (0 = MX_OK)."""
    return int(lib().mx_device_status(1 if clear else 0))
