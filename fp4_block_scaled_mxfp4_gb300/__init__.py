"""GB300 (sm_103a) MXFP4 mixture-of-experts expert FFN.

The compute path is the C-ABI library ``libmxfp4moe.so`` (hand-written CUDA: tcgen05
block-scaled grouped GEMM in MXFP4 and NVFP4, routing, MX and NVFP4 quantisers, combine,
MXFP4 / NVFP4 / FP8 dequant kernels); this package only builds it (``build.build()``)
and marshals torch tensors into its calls.
"""
from ._native import (  # noqa: F401
    MXError,
    act_quant_mxfp4,
    act_quant_mxfp8,
    act_quant_nvfp4,
    check_workspace,
    device_status,
    fp8_block_dequant_128x128,
    lib,
    library_path,
    moe_mxfp4_forward,
    moe_mxfp4_route,
    moe_mxfp4_workspace_layout,
    moe_mxfp4_workspace_size,
    moe_mxfp4w_mxfp8a_forward,
    moe_mxfp4w_mxfp8a_workspace_layout,
    moe_mxfp4w_mxfp8a_workspace_size,
    moe_nvfp4_forward,
    moe_nvfp4_workspace_layout,
    moe_nvfp4_workspace_size,
    mxfp4_dequant,
    mxfp4_gemm_bf16,
    mxfp4_scales_to_tiled,
    mxfp4_tiled_scales_bytes,
    mxfp8_mxfp4_gemm_bf16,
    nvfp4_calibrate_global,
    nvfp4_dequant,
    nvfp4_gemm_bf16,
    nvfp4_gemm_bf16_multi,
    nvfp4_scales_to_tiled,
    nvfp4_tiled_scales_bytes,
    selftest_grid_barrier_timeout,
    selftest_wait_timeout,
    status_string,
)
