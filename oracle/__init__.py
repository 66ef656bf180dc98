"""CPU oracle for the MoE expert FFN: MXFP4, NVFP4 and MXFP8 variants (test infrastructure).

This package is the plain, slow, float64 CPU statement of what the hot path computes.
It is test infrastructure: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may import or run it. The product path (the
C-ABI library and its Python binding) never imports it, and it never imports them.
"""
from .mxfp4_oracle import (  # noqa: F401
    act_quant_mxfp4,
    act_quant_mxfp8,
    bf16_bits_from_f64,
    bf16_bits_to_f64,
    e2m1_decode,
    e4m3_round_code,
    e4m3fn_decode,
    e8m0_decode,
    fp8_block_dequant_128x128,
    mxfp4_dequant,
    mxfp4_gemm_blockint,
    mxfp4_gemm_bf16,
    mxfp4_values,
    mxfp8_mxfp4_gemm_bf16,
    mxfp8_values,
    moe_combine,
    moe_forward,
    moe_mxfp8_forward,
    moe_nvfp4_forward,
    moe_l1_exact,
    moe_l2_bf16,
    moe_route,
    swiglu_bf16,
    moe_flops_per_pair,
    nvfp4_activation_global,
    nvfp4_dequant,
    nvfp4_gemm_bf16,
    nvfp4_gemm_f64,
    nvfp4_gemm_segments_bf16,
    nvfp4_quantize,
    nvfp4_values,
    unpack_nibbles,
)
