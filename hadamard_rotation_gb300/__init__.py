"""Fused Hadamard rotation + NVFP4 quantization for GB300 (sm_103a).

The compute path is libhq.so (hand-written CUDA, C ABI in include/hq.h); this package
is its Python binding.  ``synth`` draws the seeded synthetic activations.
"""
from ._lib import HQError, lib_path, load  # noqa: F401
from .api import (  # noqa: F401
    HostQuantizer,
    hq_dequant_mxfp4,
    hq_dequant_nvfp4,
    hq_quantize_nvfp4,
    hq_quantize_nvfp4_host_noalloc,
    hq_read_fault,
    hq_rot_amax,
    hq_rotate_quant_int8,
    hq_rotate_quant_mxfp4,
    hq_rotate_quant_mxfp4_ws,
    hq_rotate_quant_nvfp4,
    hq_rotate_quant_nvfp4_delayed,
    hq_rotate_quant_nvfp4_delayed_ws,
    hq_rotate_quant_nvfp4_swizzled,
    hq_rotate_quant_nvfp4_swizzled_ws,
    hq_rotate_quant_nvfp4_ws,
    hq_selftest_bounded_wait,
    hq_status_string,
    hq_swizzled_scales_bytes,
    hq_version,
    quantize_nvfp4,
)

__all__ = [
    "HQError",
    "HostQuantizer",
    "hq_dequant_mxfp4",
    "hq_dequant_nvfp4",
    "hq_quantize_nvfp4",
    "hq_quantize_nvfp4_host_noalloc",
    "hq_read_fault",
    "hq_rot_amax",
    "hq_rotate_quant_int8",
    "hq_rotate_quant_mxfp4",
    "hq_rotate_quant_mxfp4_ws",
    "hq_rotate_quant_nvfp4",
    "hq_rotate_quant_nvfp4_delayed",
    "hq_rotate_quant_nvfp4_delayed_ws",
    "hq_rotate_quant_nvfp4_swizzled",
    "hq_rotate_quant_nvfp4_swizzled_ws",
    "hq_rotate_quant_nvfp4_ws",
    "hq_selftest_bounded_wait",
    "hq_status_string",
    "hq_swizzled_scales_bytes",
    "hq_version",
    "lib_path",
    "load",
    "quantize_nvfp4",
]
