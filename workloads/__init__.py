"""Seeded synthetic inputs for the MoE expert FFN (MXFP4 and NVFP4) and its kernels.

This module is shared by the CUDA-path tests, ``bench.py`` and the oracle tests. It
holds none of the method's arithmetic: it draws random bytes, normals and routing
choices, converts the float32 draws to the bfloat16 bit patterns that are the
method's input dtype, and takes the NVFP4 activation global of a batch as its warm-up
calibration max|x| / (6 * 448), an input the method is given.
"""
from .generators import (  # noqa: F401
    CONFIGS,
    MoEInputs,
    NvMoEInputs,
    f32_to_bf16_bits,
    make_config_inputs,
    make_dequant_inputs,
    make_gemm_inputs,
    make_nvfp4_scales,
    make_moe_inputs,
    make_nvfp4_config_inputs,
    make_nvfp4_moe_inputs,
)
