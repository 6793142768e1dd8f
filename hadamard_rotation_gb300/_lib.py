"""ctypes loader for libhq.so.  No fallback: if the library is missing, calls fail loudly."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

HQ_OK = 0
HQ_ERR_NULL = 1
HQ_ERR_SHAPE = 2
HQ_ERR_ALIGN = 3
HQ_ERR_DTYPE = 4
HQ_ERR_GROUP = 5
HQ_ERR_CUDA = 6
HQ_ERR_TOO_LARGE = 7
HQ_ERR_ALIAS = 8

HQ_F32 = 0
HQ_BF16 = 1

_lock = threading.Lock()
_lib = None


class HQError(RuntimeError):
    def __init__(self, status: int, where: str, message: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f" (cudaError {cuda_error})" if status == HQ_ERR_CUDA else ""
        super().__init__(f"{where}: {message}{extra}")


def lib_path() -> str:
    return LIB


def load() -> ctypes.CDLL:
    """Load libhq.so; raise if it has not been built (there is no other implementation)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB):
            raise RuntimeError(
                f"libhq.so not found at {LIB}; build it first "
                "(python -m hadamard_rotation_gb300.build, or __graft_entry__.build())")
        lib = ctypes.CDLL(LIB)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.hq_rot_amax.argtypes = [p, i32, i64, i64, i64, i32, p, p, p]
        lib.hq_rot_amax.restype = i32
        lib.hq_rotate_quant_nvfp4.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4.restype = i32
        lib.hq_rotate_quant_nvfp4_ws.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4_ws.restype = i32
        lib.hq_quantize_nvfp4.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, p]
        lib.hq_quantize_nvfp4.restype = i32
        lib.hq_rotate_quant_nvfp4_delayed.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4_delayed.restype = i32
        lib.hq_rotate_quant_nvfp4_delayed_ws.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4_delayed_ws.restype = i32
        lib.hq_rotate_quant_nvfp4_swizzled.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4_swizzled.restype = i32
        lib.hq_rotate_quant_nvfp4_swizzled_ws.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, p]
        lib.hq_rotate_quant_nvfp4_swizzled_ws.restype = i32
        lib.hq_swizzled_scales_bytes.argtypes = [i64, i64]
        lib.hq_swizzled_scales_bytes.restype = i64
        lib.hq_rotate_quant_mxfp4.argtypes = [p, i32, i64, i64, i64, i32, p, p, p]
        lib.hq_rotate_quant_mxfp4.restype = i32
        lib.hq_rotate_quant_mxfp4_ws.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p]
        lib.hq_rotate_quant_mxfp4_ws.restype = i32
        lib.hq_dequant_mxfp4.argtypes = [p, p, i64, i64, i32, i32, p, p]
        lib.hq_dequant_mxfp4.restype = i32
        lib.hq_rotate_quant_int8.argtypes = [p, i32, i64, i64, i64, i32, p, p, p]
        lib.hq_rotate_quant_int8.restype = i32
        lib.hq_dequant_nvfp4.argtypes = [p, p, p, i64, i64, i32, i32, p, p]
        lib.hq_dequant_nvfp4.restype = i32
        lib.hq_status_string.argtypes = [i32]
        lib.hq_status_string.restype = ctypes.c_char_p
        lib.hq_last_cuda_error.argtypes = []
        lib.hq_last_cuda_error.restype = i32
        sz = ctypes.c_size_t
        lib.hq_host_pipeline_workspace_bytes.argtypes = [i64, i64, i32]
        lib.hq_host_pipeline_workspace_bytes.restype = sz
        lib.hq_host_pipeline_create.argtypes = [i64, i64, i32, i32, p, sz, ctypes.POINTER(p)]
        lib.hq_host_pipeline_create.restype = i32
        lib.hq_host_pipeline_submit.argtypes = [p, p, p, p, p]
        lib.hq_host_pipeline_submit.restype = i32
        lib.hq_host_pipeline_wait.argtypes = [p]
        lib.hq_host_pipeline_wait.restype = i32
        lib.hq_host_pipeline_destroy.argtypes = [p]
        lib.hq_host_pipeline_destroy.restype = i32
        lib.hq_host_pipeline_inject_failure.argtypes = [p, i32]
        lib.hq_host_pipeline_inject_failure.restype = i32
        lib.hq_read_fault.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        lib.hq_read_fault.restype = i32
        lib.hq_quantize_nvfp4_host_noalloc.argtypes = [p, i32, i64, i64, i32, p, p, p, p]
        lib.hq_quantize_nvfp4_host_noalloc.restype = i32
        lib.hq_selftest_bounded_wait.argtypes = [i32, p]
        lib.hq_selftest_bounded_wait.restype = i32
        lib.hq_version.argtypes = []
        lib.hq_version.restype = i32
        _lib = lib
        return lib


def check(status: int, where: str) -> None:
    if status != HQ_OK:
        lib = load()
        msg = lib.hq_status_string(status).decode()
        raise HQError(status, where, msg, lib.hq_last_cuda_error())
