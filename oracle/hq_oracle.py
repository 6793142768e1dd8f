"""ctypes wrapper over the C++ oracle (``hq_oracle.cpp``).

Test infrastructure only.  Inputs and outputs are numpy arrays on the host; the
oracle never touches a GPU and shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hq_oracle.cpp")
_LIB = os.path.join(_HERE, "libhq_oracle.so")

DT_F32 = 0
DT_BF16 = 1

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (scalar fp32, no contraction, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
            lib.hqo_rot_amax.argtypes = [p, i32, i64, i64, i64, i32, p, p, i32]
            lib.hqo_rot_amax.restype = i32
            lib.hqo_quantize.argtypes = [p, i32, i64, i64, i64, i32, p, p, p, p, p, i32]
            lib.hqo_quantize.restype = i32
            lib.hqo_dequant.argtypes = [p, p, ctypes.c_float, i64, i64, i32, i32, p, i32]
            lib.hqo_dequant.restype = i32
            lib.hqo_rotate.argtypes = [p, i64, i32, p]
            lib.hqo_rotate.restype = i32
            lib.hqo_e2m1_codes.argtypes = [p, i64, p]
            lib.hqo_e2m1_codes.restype = None
            lib.hqo_e2m1_codes_bits.argtypes = [u32, i64, p, i32]
            lib.hqo_e2m1_codes_bits.restype = None
            lib.hqo_e4m3_codes.argtypes = [p, i64, p, i32]
            lib.hqo_e4m3_codes.restype = None
            lib.hqo_e4m3_codes_bits.argtypes = [u32, i64, p, i32]
            lib.hqo_e4m3_codes_bits.restype = None
            lib.hqo_e4m3_values.argtypes = [p, i64, p]
            lib.hqo_e4m3_values.restype = None
            lib.hqo_int8_rotate.argtypes = [p, i64, i32, p]
            lib.hqo_int8_rotate.restype = i32
            lib.hqo_rotate_quant_int8.argtypes = [p, i32, i64, i64, i64, i32, p, p, i32]
            lib.hqo_rotate_quant_int8.restype = i32
            lib.hqo_quantize_mxfp4.argtypes = [p, i32, i64, i64, i64, i32, p, p, i32]
            lib.hqo_quantize_mxfp4.restype = i32
            lib.hqo_dequant_mxfp4.argtypes = [p, p, i64, i64, i32, i32, p, i32]
            lib.hqo_dequant_mxfp4.restype = i32
            lib.hqo_global_scale.argtypes = [ctypes.c_float]
            lib.hqo_global_scale.restype = ctypes.c_float
            _lib = lib
    return _lib


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _x_dtype(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return DT_F32
    if x.dtype == np.uint16:  # bf16 bit patterns
        return DT_BF16
    raise TypeError(f"oracle input must be float32 or uint16 (bf16 bits), got {x.dtype}")


def _check2d(x: np.ndarray):
    if x.ndim != 2:
        raise ValueError("x must be 2-D [M, K]")
    if x.strides[1] != x.itemsize:
        raise ValueError("rows of x must be contiguous")
    M, K = x.shape
    ldx = x.strides[0] // x.itemsize if M > 1 else K
    return M, K, ldx


def rot_amax(x: np.ndarray, group: int, want_y: bool = False, nthreads: int | None = None):
    """Return (amax, y or None); y is the fp32 rotated tensor [M, K]."""
    lib = _load()
    M, K, ldx = _check2d(x)
    amax = np.zeros(1, np.float32)
    y = np.empty((M, K), np.float32) if want_y else None
    rc = lib.hqo_rot_amax(_ptr(x), _x_dtype(x), M, K, ldx, group, _ptr(amax),
                          _ptr(y) if y is not None else None, _threads(nthreads))
    if rc:
        raise ValueError("hqo_rot_amax: bad arguments")
    return amax[0], y


def quantize(x: np.ndarray, group: int, amax: float | None = None, nthreads: int | None = None):
    """Return (q [M,K/2] u8, scales [M,K/16] u8, amax f32, s_global f32)."""
    lib = _load()
    M, K, ldx = _check2d(x)
    q = np.empty((M, K // 2), np.uint8)
    s = np.empty((M, K // 16), np.uint8)
    amax_out = np.zeros(1, np.float32)
    sg = np.zeros(1, np.float32)
    amax_in = np.array([amax], np.float32) if amax is not None else None
    rc = lib.hqo_quantize(_ptr(x), _x_dtype(x), M, K, ldx, group,
                          _ptr(amax_in) if amax_in is not None else None,
                          _ptr(q), _ptr(s), _ptr(amax_out), _ptr(sg), _threads(nthreads))
    if rc:
        raise ValueError("hqo_quantize: bad arguments")
    return q, s, amax_out[0], sg[0]


def dequant(q: np.ndarray, s: np.ndarray, s_global: float, group: int, unrotate: bool,
            nthreads: int | None = None) -> np.ndarray:
    lib = _load()
    M = q.shape[0]
    K = q.shape[1] * 2
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    out = np.empty((M, K), np.float32)
    rc = lib.hqo_dequant(_ptr(q), _ptr(s), ctypes.c_float(s_global), M, K, group,
                         1 if unrotate else 0, _ptr(out), _threads(nthreads))
    if rc:
        raise ValueError("hqo_dequant: bad arguments")
    return out


def rotate(x: np.ndarray, group: int) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty_like(x)
    if lib.hqo_rotate(_ptr(x), x.size, group, _ptr(out)):
        raise ValueError("hqo_rotate: bad arguments")
    return out


def e2m1_codes(v: np.ndarray) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib.hqo_e2m1_codes(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_codes_bits(first: int, count: int, nthreads: int | None = None) -> np.ndarray:
    lib = _load()
    out = np.empty(count, np.uint8)
    lib.hqo_e2m1_codes_bits(first, count, _ptr(out), _threads(nthreads))
    return out


def e4m3_codes(v: np.ndarray, nthreads: int | None = None) -> np.ndarray:
    lib = _load()
    v = np.ascontiguousarray(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib.hqo_e4m3_codes(_ptr(v), v.size, _ptr(out), _threads(nthreads))
    return out


def e4m3_codes_bits(first: int, count: int, nthreads: int | None = None) -> np.ndarray:
    lib = _load()
    out = np.empty(count, np.uint8)
    lib.hqo_e4m3_codes_bits(first, count, _ptr(out), _threads(nthreads))
    return out


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    codes = np.ascontiguousarray(codes, np.uint8)
    out = np.empty(codes.shape, np.float32)
    lib.hqo_e4m3_values(_ptr(codes), codes.size, _ptr(out))
    return out


def global_scale(amax: float) -> float:
    return float(_load().hqo_global_scale(ctypes.c_float(amax)))


def int8_rotate(x: np.ndarray, group: int) -> np.ndarray:
    """y = x . R_G (regular Hadamard) on every run of `group` values."""
    lib = _load()
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty_like(x)
    if lib.hqo_int8_rotate(_ptr(x), x.size, group, _ptr(out)):
        raise ValueError("hqo_int8_rotate: bad arguments")
    return out


def rotate_quant_int8(x: np.ndarray, group: int, nthreads: int | None = None):
    """Return (q int8 [M, K], scales float32 [M])."""
    lib = _load()
    M, K, ldx = _check2d(x)
    q = np.empty((M, K), np.int8)
    sc = np.empty(M, np.float32)
    rc = lib.hqo_rotate_quant_int8(_ptr(x), _x_dtype(x), M, K, ldx, group, _ptr(q), _ptr(sc),
                                   _threads(nthreads))
    if rc:
        raise ValueError("hqo_rotate_quant_int8: bad arguments")
    return q, sc


def quantize_mxfp4(x: np.ndarray, group: int, nthreads: int | None = None):
    """Return (q [M, K/2] u8, scales [M, K/32] E8M0 u8)."""
    lib = _load()
    M, K, ldx = _check2d(x)
    q = np.empty((M, K // 2), np.uint8)
    s = np.empty((M, K // 32), np.uint8)
    rc = lib.hqo_quantize_mxfp4(_ptr(x), _x_dtype(x), M, K, ldx, group, _ptr(q), _ptr(s),
                                _threads(nthreads))
    if rc:
        raise ValueError("hqo_quantize_mxfp4: bad arguments")
    return q, s


def dequant_mxfp4(q: np.ndarray, s: np.ndarray, group: int, unrotate: bool,
                  nthreads: int | None = None) -> np.ndarray:
    lib = _load()
    M, K = q.shape[0], q.shape[1] * 2
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    out = np.empty((M, K), np.float32)
    if lib.hqo_dequant_mxfp4(_ptr(q), _ptr(s), M, K, group, 1 if unrotate else 0, _ptr(out),
                             _threads(nthreads)):
        raise ValueError("hqo_dequant_mxfp4: bad arguments")
    return out


def swizzle_scales(s: np.ndarray) -> np.ndarray:
    """Row-major block scales [M, K/16] -> the swizzled tile layout of block-scaled NVFP4 GEMMs.

    "A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §6 "From interpreter to hardware"
    (Layout): GEMM consumers take the scales in a swizzled tiled layout, not spelled out on the
    page.  Reading: cuBLASLt's layout for 16-element block scales.  The matrix is padded with
    zeros to R = round_up(M, 128) rows and C = round_up(K/16, 4) columns and cut into tiles of
    128 rows x 4 columns; tile (i, j) is the 512 bytes at (i * C/4 + j) * 512, and inside it row
    r, column c is the byte (r % 32) * 16 + (r / 32) * 4 + c.  Pinned on the GPU by feeding the
    library's output to cuBLASLt's NVFP4 GEMM (tests/test_gpu_swizzle.py).
    """
    s = np.ascontiguousarray(s, np.uint8)
    M, C0 = s.shape
    R = -(-M // 128) * 128
    C = -(-C0 // 4) * 4
    out = np.zeros(R * C, np.uint8)
    for r in range(M):
        i, rr = divmod(r, 128)
        for c in range(C0):
            j, cc = divmod(c, 4)
            out[(i * (C // 4) + j) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc] = s[r, c]
    return out


def unswizzle_scales(buf: np.ndarray, M: int, C0: int) -> np.ndarray:
    """Inverse of swizzle_scales: the [M, C0] row-major scales held in a swizzled buffer."""
    C = -(-C0 // 4) * 4
    out = np.empty((M, C0), np.uint8)
    for r in range(M):
        i, rr = divmod(r, 128)
        for c in range(C0):
            j, cc = divmod(c, 4)
            out[r, c] = buf[(i * (C // 4) + j) * 512 + (rr % 32) * 16 + (rr // 32) * 4 + cc]
    return out
