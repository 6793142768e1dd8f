"""CPU oracle for the fused Hadamard rotation + NVFP4 quantization.

Test infrastructure only: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  See ``hq_oracle.cpp`` for
the definition and its sources.
"""
from .hq_oracle import (  # noqa: F401
    DT_BF16,
    DT_F32,
    build,
    dequant,
    dequant_mxfp4,
    e2m1_codes,
    e2m1_codes_bits,
    e4m3_codes,
    e4m3_codes_bits,
    e4m3_values,
    global_scale,
    int8_rotate,
    lib_path,
    quantize,
    quantize_mxfp4,
    rot_amax,
    rotate,
    rotate_quant_int8,
    swizzle_scales,
    unswizzle_scales,
)
