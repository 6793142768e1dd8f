"""Python binding of libhq: the C ABI calls under the same names, over torch tensors.

Argument marshalling only.  Every step of the rotation and quantization runs in the CUDA
kernels of libhq.so; torch provides device memory, streams and pinned host buffers.
Inputs must be CUDA tensors: there is no CPU path.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import HQ_BF16, HQ_F32, check

_DTYPES = {torch.float32: HQ_F32, torch.bfloat16: HQ_BF16}


def _stream_handle(stream: torch.cuda.Stream | None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _x_args(x: torch.Tensor):
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError("x must be a CUDA tensor (libhq has no CPU path)")
    if x.dim() != 2:
        raise ValueError("x must be 2-D [M, K]")
    if x.dtype not in _DTYPES:
        raise ValueError(f"x must be float32 or bfloat16, got {x.dtype}")
    M, K = x.shape
    if K > 1 and x.stride(1) != 1:
        raise ValueError("rows of x must be contiguous (stride(1) == 1)")
    ldx = x.stride(0) if M > 1 else K
    return _DTYPES[x.dtype], M, K, ldx


def _need(t: torch.Tensor | None, shape, dtype, device, name):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous() or t.device != device:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")
    return t


def hq_rot_amax(x: torch.Tensor, group: int, amax: torch.Tensor | None = None,
                y: torch.Tensor | None = None,
                stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Pass 1: max |x . H_G / sqrt(G)| into a 1-element float32 device tensor.

    ``y`` (optional, float32 [M, K]) receives the rotated tensor.
    """
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    if y is not None:
        y = _need(y, (M, K), torch.float32, x.device, "y")
    check(_lib.load().hq_rot_amax(_ptr(x), dt, M, K, ldx, group, _ptr(amax), _ptr(y),
                                  _stream_handle(stream)), "hq_rot_amax")
    return amax


def hq_rotate_quant_nvfp4(x: torch.Tensor, group: int, amax: torch.Tensor,
                          q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                          s_global: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None):
    """Pass 2: (q uint8 [M, K/2], scales uint8 [M, K/16] E4M3 bits, s_global float32 [1])."""
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    check(_lib.load().hq_rotate_quant_nvfp4(_ptr(x), dt, M, K, ldx, group, _ptr(amax), _ptr(q),
                                            _ptr(scales), _ptr(s_global), _stream_handle(stream)),
          "hq_rotate_quant_nvfp4")
    return q, scales, s_global


def hq_dequant_nvfp4(q: torch.Tensor, scales: torch.Tensor, s_global: torch.Tensor, group: int,
                     unrotate: bool, out: torch.Tensor | None = None,
                     stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Round trip: float32 [M, K] = codes * (s_block * s_global), optionally un-rotated."""
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor (libhq has no CPU path)")
    M, K2 = q.shape
    K = 2 * K2
    q = _need(q, (M, K2), torch.uint8, q.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, q.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, q.device, "s_global")
    out = _need(out, (M, K), torch.float32, q.device, "out")
    check(_lib.load().hq_dequant_nvfp4(_ptr(q), _ptr(scales), _ptr(s_global), M, K, group,
                                       1 if unrotate else 0, _ptr(out), _stream_handle(stream)),
          "hq_dequant_nvfp4")
    return out


def quantize_nvfp4(x: torch.Tensor, group: int, stream: torch.cuda.Stream | None = None):
    """Both passes: (q, scales, s_global, amax), all on x's device."""
    amax = hq_rot_amax(x, group, stream=stream)
    q, s, sg = hq_rotate_quant_nvfp4(x, group, amax, stream=stream)
    return q, s, sg, amax


class HostQuantizer:
    """Quantize host tensors: pinned host -> device, both passes, device -> pinned host.

    Device buffers and pinned outputs are allocated once here; each call then enqueues
    one host-to-device copy of x, the two kernels and the device-to-host copies of the
    codes, scales and s_global on ``stream``.
    """

    def __init__(self, M: int, K: int, dtype: torch.dtype, group: int,
                 device: torch.device | str = "cuda", stream: torch.cuda.Stream | None = None):
        self.M, self.K, self.group = M, K, group
        self.device = torch.device(device)
        self.stream = stream
        self.x_dev = torch.empty((M, K), dtype=dtype, device=self.device)
        self.amax = torch.empty(1, dtype=torch.float32, device=self.device)
        self.q_dev = torch.empty((M, K // 2), dtype=torch.uint8, device=self.device)
        self.s_dev = torch.empty((M, K // 16), dtype=torch.uint8, device=self.device)
        self.sg_dev = torch.empty(1, dtype=torch.float32, device=self.device)
        self.q_host = torch.empty((M, K // 2), dtype=torch.uint8, pin_memory=True)
        self.s_host = torch.empty((M, K // 16), dtype=torch.uint8, pin_memory=True)
        self.sg_host = torch.empty(1, dtype=torch.float32, pin_memory=True)

    @property
    def h2d_bytes(self) -> int:
        return self.x_dev.numel() * self.x_dev.element_size()

    @property
    def d2h_bytes(self) -> int:
        return self.q_host.numel() + self.s_host.numel() + 4

    def enqueue(self, x_host: torch.Tensor) -> None:
        """Enqueue one quantization of the pinned host tensor ``x_host`` (no host sync)."""
        s = self.stream if self.stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self.x_dev.copy_(x_host, non_blocking=True)
            hq_rot_amax(self.x_dev, self.group, amax=self.amax, stream=s)
            hq_rotate_quant_nvfp4(self.x_dev, self.group, self.amax, q=self.q_dev,
                                  scales=self.s_dev, s_global=self.sg_dev, stream=s)
            self.q_host.copy_(self.q_dev, non_blocking=True)
            self.s_host.copy_(self.s_dev, non_blocking=True)
            self.sg_host.copy_(self.sg_dev, non_blocking=True)

    def __call__(self, x_host: torch.Tensor):
        self.enqueue(x_host)
        s = self.stream if self.stream is not None else torch.cuda.current_stream(self.device)
        s.synchronize()
        return self.q_host, self.s_host, float(self.sg_host[0])
