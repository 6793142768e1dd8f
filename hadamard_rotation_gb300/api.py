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


def _stream_handle(stream: torch.cuda.Stream | None,
                   device: torch.device | None = None) -> ctypes.c_void_p:
    """The cudaStream_t to pass: ``stream``, or the current stream of ``device`` (default: the
    current device).  A given stream must belong to ``device``."""
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if device is not None and stream.device != device:
        raise ValueError(f"stream is on {stream.device}, the tensors on {device}")
    return ctypes.c_void_p(stream.cuda_stream)


def _call(device: torch.device, name: str, *args, stream: torch.cuda.Stream | None = None) -> None:
    """Call the C entry point ``name`` with ``device`` current (the library launches on the
    current device), on ``stream`` or that device's current stream; raise on a non-OK status."""
    with torch.cuda.device(device):
        check(getattr(_lib.load(), name)(*args, _stream_handle(stream, device)), name)


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
    _call(x.device, "hq_rot_amax", _ptr(x), dt, M, K, ldx, group, _ptr(amax), _ptr(y),
          stream=stream)
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
    _call(x.device, "hq_rotate_quant_nvfp4", _ptr(x), dt, M, K, ldx, group, _ptr(amax), _ptr(q),
          _ptr(scales), _ptr(s_global), stream=stream)
    return q, scales, s_global


# The workspaces of hq_quantize_nvfp4 and the _ws entry points kept by this binding, one
# per (device, stream).
_WORKSPACES: dict[tuple[int, int], torch.Tensor] = {}
HQ_QUANTIZE_WORKSPACE_WORDS = 288


def _workspace(device: torch.device, stream: torch.cuda.Stream | None) -> torch.Tensor:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index if device.index is not None else torch.cuda.current_device(), s.cuda_stream)
    w = _WORKSPACES.get(key)
    if w is None:
        w = torch.zeros(HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=device)
        _WORKSPACES[key] = w
    return w


def hq_rotate_quant_nvfp4_ws(x: torch.Tensor, group: int, amax: torch.Tensor,
                             q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                             s_global: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None,
                             stream: torch.cuda.Stream | None = None):
    """Pass 2 as hq_rotate_quant_nvfp4, with the tiles handed to the warps at run time from the
    counters in ``workspace`` (int32 [HQ_QUANTIZE_WORKSPACE_WORDS], zero before first use;
    default: the one this binding keeps per device and stream)."""
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    workspace = _workspace(x.device, stream) if workspace is None else _need(
        workspace, (HQ_QUANTIZE_WORKSPACE_WORDS,), torch.int32, x.device, "workspace")
    _call(x.device, "hq_rotate_quant_nvfp4_ws", _ptr(x), dt, M, K, ldx, group, _ptr(amax),
          _ptr(q), _ptr(scales), _ptr(s_global), _ptr(workspace), stream=stream)
    return q, scales, s_global


def hq_quantize_nvfp4(x: torch.Tensor, group: int, amax: torch.Tensor | None = None,
                      q: torch.Tensor | None = None, scales: torch.Tensor | None = None,
                      s_global: torch.Tensor | None = None, use_workspace: bool = True,
                      workspace: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None):
    """Both passes in one call: (q, scales, s_global, amax), as hq_rot_amax then
    hq_rotate_quant_nvfp4.  With ``use_workspace`` (default) the call passes a workspace (int32
    [HQ_QUANTIZE_WORKSPACE_WORDS], zero before first use; default: one this binding keeps per
    device and stream): pass 1 reduces the amax into it without a memset and pass 2 takes its
    tiles at run time; without, the plain hq_rot_amax then hq_rotate_quant_nvfp4."""
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    if use_workspace:
        workspace = _workspace(x.device, stream) if workspace is None else _need(
            workspace, (HQ_QUANTIZE_WORKSPACE_WORDS,), torch.int32, x.device, "workspace")
    else:
        workspace = None
    _call(x.device, "hq_quantize_nvfp4", _ptr(x), dt, M, K, ldx, group, _ptr(amax), _ptr(q),
          _ptr(scales), _ptr(s_global), _ptr(workspace), stream=stream)
    return q, scales, s_global, amax


def hq_swizzled_scales_bytes(M: int, K: int) -> int:
    """Bytes of the swizzled scale buffer for an [M, K] tensor (128-row x 4-column tiles)."""
    n = _lib.load().hq_swizzled_scales_bytes(M, K)
    if n < 0:
        raise ValueError("hq_swizzled_scales_bytes: M, K must be >= 0 and K a multiple of 16")
    return n


def hq_rotate_quant_nvfp4_swizzled(x: torch.Tensor, group: int, amax: torch.Tensor,
                                   q: torch.Tensor | None = None,
                                   scales: torch.Tensor | None = None,
                                   s_global: torch.Tensor | None = None,
                                   stream: torch.cuda.Stream | None = None):
    """Pass 2 with the block scales in the swizzled tile layout of block-scaled NVFP4 GEMMs:
    (q uint8 [M, K/2], scales uint8 [hq_swizzled_scales_bytes(M, K)], s_global float32 [1]).
    Every byte of ``scales`` is written, padding entries as 0."""
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    n = hq_swizzled_scales_bytes(M, K)
    scales = _need(scales, (n,), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    _call(x.device, "hq_rotate_quant_nvfp4_swizzled", _ptr(x), dt, M, K, ldx, group, _ptr(amax),
          _ptr(q), _ptr(scales), _ptr(s_global), stream=stream)
    return q, scales, s_global


def hq_rotate_quant_nvfp4_swizzled_ws(x: torch.Tensor, group: int, amax: torch.Tensor,
                                      q: torch.Tensor | None = None,
                                      scales: torch.Tensor | None = None,
                                      s_global: torch.Tensor | None = None,
                                      workspace: torch.Tensor | None = None,
                                      stream: torch.cuda.Stream | None = None):
    """hq_rotate_quant_nvfp4_swizzled with its units of work handed to the warps at run time from
    the counters in ``workspace`` (as hq_rotate_quant_nvfp4_ws; default: the one this binding
    keeps per device and stream)."""
    dt, M, K, ldx = _x_args(x)
    amax = _need(amax, (1,), torch.float32, x.device, "amax")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (hq_swizzled_scales_bytes(M, K),), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    workspace = _workspace(x.device, stream) if workspace is None else _need(
        workspace, (HQ_QUANTIZE_WORKSPACE_WORDS,), torch.int32, x.device, "workspace")
    _call(x.device, "hq_rotate_quant_nvfp4_swizzled_ws", _ptr(x), dt, M, K, ldx, group,
          _ptr(amax), _ptr(q), _ptr(scales), _ptr(s_global), _ptr(workspace), stream=stream)
    return q, scales, s_global


def hq_rotate_quant_nvfp4_delayed(x: torch.Tensor, group: int, amax_prev: torch.Tensor,
                                  amax_next: torch.Tensor | None = None,
                                  q: torch.Tensor | None = None,
                                  scales: torch.Tensor | None = None,
                                  s_global: torch.Tensor | None = None,
                                  stream: torch.cuda.Stream | None = None):
    """Single pass with a delayed amax: quantize with ``amax_prev`` and reduce this tensor's
    amax into ``amax_next``.  Returns (q, scales, s_global, amax_next)."""
    dt, M, K, ldx = _x_args(x)
    amax_prev = _need(amax_prev, (1,), torch.float32, x.device, "amax_prev")
    amax_next = _need(amax_next, (1,), torch.float32, x.device, "amax_next")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    _call(x.device, "hq_rotate_quant_nvfp4_delayed", _ptr(x), dt, M, K, ldx, group,
          _ptr(amax_prev), _ptr(amax_next), _ptr(q), _ptr(scales), _ptr(s_global), stream=stream)
    return q, scales, s_global, amax_next


def hq_rotate_quant_nvfp4_delayed_ws(x: torch.Tensor, group: int, amax_prev: torch.Tensor,
                                     amax_next: torch.Tensor | None = None,
                                     q: torch.Tensor | None = None,
                                     scales: torch.Tensor | None = None,
                                     s_global: torch.Tensor | None = None,
                                     workspace: torch.Tensor | None = None,
                                     stream: torch.cuda.Stream | None = None):
    """hq_rotate_quant_nvfp4_delayed with a workspace (as hq_rotate_quant_nvfp4_ws; default: the
    one this binding keeps per device and stream): tiles handed out at run time, and the next
    amax reduced in the workspace instead of after a memset.  Returns (q, scales, s_global,
    amax_next)."""
    dt, M, K, ldx = _x_args(x)
    amax_prev = _need(amax_prev, (1,), torch.float32, x.device, "amax_prev")
    amax_next = _need(amax_next, (1,), torch.float32, x.device, "amax_next")
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 16), torch.uint8, x.device, "scales")
    s_global = _need(s_global, (1,), torch.float32, x.device, "s_global")
    workspace = _workspace(x.device, stream) if workspace is None else _need(
        workspace, (HQ_QUANTIZE_WORKSPACE_WORDS,), torch.int32, x.device, "workspace")
    _call(x.device, "hq_rotate_quant_nvfp4_delayed_ws", _ptr(x), dt, M, K, ldx, group,
          _ptr(amax_prev), _ptr(amax_next), _ptr(q), _ptr(scales), _ptr(s_global), _ptr(workspace),
          stream=stream)
    return q, scales, s_global, amax_next


def hq_rotate_quant_mxfp4(x: torch.Tensor, group: int, q: torch.Tensor | None = None,
                          scales: torch.Tensor | None = None,
                          stream: torch.cuda.Stream | None = None):
    """MXFP4: (q uint8 [M, K/2], scales uint8 [M, K/32] E8M0 bytes); one pass over x."""
    dt, M, K, ldx = _x_args(x)
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 32), torch.uint8, x.device, "scales")
    _call(x.device, "hq_rotate_quant_mxfp4", _ptr(x), dt, M, K, ldx, group, _ptr(q), _ptr(scales),
          stream=stream)
    return q, scales


def hq_rotate_quant_mxfp4_ws(x: torch.Tensor, group: int, q: torch.Tensor | None = None,
                             scales: torch.Tensor | None = None,
                             workspace: torch.Tensor | None = None,
                             stream: torch.cuda.Stream | None = None):
    """MXFP4 as hq_rotate_quant_mxfp4, with the tiles handed to the warps at run time from the
    counters in ``workspace`` (as hq_rotate_quant_nvfp4_ws; default: the one this binding keeps
    per device and stream)."""
    dt, M, K, ldx = _x_args(x)
    q = _need(q, (M, K // 2), torch.uint8, x.device, "q")
    scales = _need(scales, (M, K // 32), torch.uint8, x.device, "scales")
    workspace = _workspace(x.device, stream) if workspace is None else _need(
        workspace, (HQ_QUANTIZE_WORKSPACE_WORDS,), torch.int32, x.device, "workspace")
    _call(x.device, "hq_rotate_quant_mxfp4_ws", _ptr(x), dt, M, K, ldx, group, _ptr(q),
          _ptr(scales), _ptr(workspace), stream=stream)
    return q, scales


def hq_dequant_mxfp4(q: torch.Tensor, scales: torch.Tensor, group: int, unrotate: bool,
                     out: torch.Tensor | None = None,
                     stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """MXFP4 round trip: float32 [M, K] = codes * 2^(byte - 127), optionally un-rotated."""
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor (libhq has no CPU path)")
    M, K2 = q.shape
    K = 2 * K2
    q = _need(q, (M, K2), torch.uint8, q.device, "q")
    scales = _need(scales, (M, K // 32), torch.uint8, q.device, "scales")
    out = _need(out, (M, K), torch.float32, q.device, "out")
    _call(q.device, "hq_dequant_mxfp4", _ptr(q), _ptr(scales), M, K, group, 1 if unrotate else 0,
          _ptr(out), stream=stream)
    return out


def hq_rotate_quant_int8(x: torch.Tensor, group: int, q: torch.Tensor | None = None,
                         scales: torch.Tensor | None = None,
                         stream: torch.cuda.Stream | None = None):
    """INT8 per-token rotate-quant: (q int8 [M, K], scales float32 [M])."""
    dt, M, K, ldx = _x_args(x)
    q = _need(q, (M, K), torch.int8, x.device, "q")
    scales = _need(scales, (M,), torch.float32, x.device, "scales")
    _call(x.device, "hq_rotate_quant_int8", _ptr(x), dt, M, K, ldx, group, _ptr(q), _ptr(scales),
          stream=stream)
    return q, scales


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
    _call(q.device, "hq_dequant_nvfp4", _ptr(q), _ptr(scales), _ptr(s_global), M, K, group,
          1 if unrotate else 0, _ptr(out), stream=stream)
    return out


def quantize_nvfp4(x: torch.Tensor, group: int, stream: torch.cuda.Stream | None = None):
    """Both passes: (q, scales, s_global, amax), all on x's device (hq_quantize_nvfp4)."""
    return hq_quantize_nvfp4(x, group, stream=stream)


def hq_quantize_nvfp4_host_noalloc(x_host: torch.Tensor, group: int,
                                   q_host: torch.Tensor | None = None,
                                   s_host: torch.Tensor | None = None,
                                   sg_host: torch.Tensor | None = None,
                                   stream: torch.cuda.Stream | None = None):
    """One host tensor through both passes with no device allocation (the library's fixed
    staging array; see include/hq.h for its size limit and sharing rules).  Outputs default to
    new pinned host tensors; they are complete once ``stream`` (default: current) is
    synchronised.  Returns (q_host, s_host, sg_host)."""
    if not isinstance(x_host, torch.Tensor) or x_host.is_cuda or x_host.dim() != 2 \
            or x_host.dtype not in _DTYPES or not x_host.is_contiguous():
        raise ValueError("x_host must be a contiguous 2-D float32 or bfloat16 host tensor")
    M, K = x_host.shape
    outs = []
    for t, shape, dt, name in ((q_host, (M, K // 2), torch.uint8, "q_host"),
                               (s_host, (M, K // 16), torch.uint8, "s_host"),
                               (sg_host, (1,), torch.float32, "sg_host")):
        if t is None:
            t = torch.empty(shape, dtype=dt, pin_memory=True)
        elif t.is_cuda or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host {dt} tensor {shape}")
        outs.append(t)
    check(_lib.load().hq_quantize_nvfp4_host_noalloc(
        _ptr(x_host), _DTYPES[x_host.dtype], M, K, group, _ptr(outs[0]), _ptr(outs[1]),
        _ptr(outs[2]), _stream_handle(stream)), "hq_quantize_nvfp4_host_noalloc")
    return tuple(outs)


def hq_read_fault(clear: bool = False) -> int:
    """The device fault word (waits for the device to be idle); bit 0: a kernel's bounded wait
    for one of its own tile copies ran out.  ``clear`` resets it after reading, and zeroes the
    workspaces this binding keeps on the current device (a fault can leave one non-zero)."""
    v = ctypes.c_uint(0)
    check(_lib.load().hq_read_fault(ctypes.byref(v), 1 if clear else 0), "hq_read_fault")
    if clear:
        dev = torch.cuda.current_device()
        for (d, _), w in _WORKSPACES.items():
            if d == dev:
                w.zero_()
        torch.cuda.synchronize()
    return v.value


def hq_selftest_bounded_wait(unit: int = 0, stream: torch.cuda.Stream | None = None) -> None:
    """Enqueue the bounded-wait self-test (one warp waits on a barrier nothing completes, gives
    up after about a second and records bit 0 of the fault word).  unit 0: the NVFP4 / MXFP4
    kernels' translation unit, 1: the INT8 kernel's."""
    check(_lib.load().hq_selftest_bounded_wait(unit, _stream_handle(stream)), "hq_selftest_bounded_wait")


def hq_version() -> int:
    return int(_lib.load().hq_version())


def hq_status_string(status: int) -> str:
    return _lib.load().hq_status_string(status).decode()


class HostQuantizer:
    """Quantize tensors that live in pinned host memory, through the library's host pipeline.

    The pipeline (hq_host_pipeline_* in include/hq.h) copies x to the device, runs both passes
    and copies the codes, scales and s_global back.  Consecutive submissions overlap: the input
    copy of one runs while the previous one computes and copies its results back.  Its device
    workspace (two buffer sets) is allocated here with torch; the library allocates none.
    """

    def __init__(self, M: int, K: int, dtype: torch.dtype, group: int,
                 device: torch.device | str = "cuda"):
        if dtype not in _DTYPES:
            raise ValueError(f"dtype must be float32 or bfloat16, got {dtype}")
        self.M, self.K, self.group, self.dtype = M, K, group, dtype
        self.device = torch.device(device)
        lib = _lib.load()
        dt = _DTYPES[dtype]
        nbytes = lib.hq_host_pipeline_workspace_bytes(M, K, dt)
        if nbytes == 0:
            raise ValueError(f"invalid sizes for the host pipeline: M={M}, K={K}")
        self.work = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        handle = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            check(lib.hq_host_pipeline_create(M, K, dt, group, _ptr(self.work), nbytes,
                                              ctypes.byref(handle)), "hq_host_pipeline_create")
        self._handle = handle
        self.q_host = torch.empty((M, K // 2), dtype=torch.uint8, pin_memory=True)
        self.s_host = torch.empty((M, K // 16), dtype=torch.uint8, pin_memory=True)
        self.sg_host = torch.empty(1, dtype=torch.float32, pin_memory=True)

    @property
    def h2d_bytes(self) -> int:
        return self.M * self.K * (2 if self.dtype == torch.bfloat16 else 4)

    @property
    def d2h_bytes(self) -> int:
        return self.M * self.K // 2 + self.M * self.K // 16 + 4

    def submit(self, x_host: torch.Tensor, q_host: torch.Tensor | None = None,
               s_host: torch.Tensor | None = None, sg_host: torch.Tensor | None = None) -> None:
        """Enqueue one quantization of ``x_host``; outputs go to the given host tensors (default:
        this object's pinned buffers).  Every buffer must stay untouched until wait()."""
        if x_host.is_cuda or x_host.dtype != self.dtype or tuple(x_host.shape) != (self.M, self.K) \
                or not x_host.is_contiguous():
            raise ValueError(f"x_host must be a contiguous host {self.dtype} tensor [{self.M}, {self.K}]")
        q_host = self.q_host if q_host is None else q_host
        s_host = self.s_host if s_host is None else s_host
        sg_host = self.sg_host if sg_host is None else sg_host
        for t, shape, dt, name in ((q_host, (self.M, self.K // 2), torch.uint8, "q_host"),
                                   (s_host, (self.M, self.K // 16), torch.uint8, "s_host"),
                                   (sg_host, (1,), torch.float32, "sg_host")):
            if t.is_cuda or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous host {dt} tensor {shape}")
        check(_lib.load().hq_host_pipeline_submit(self._handle, _ptr(x_host), _ptr(q_host),
                                                  _ptr(s_host), _ptr(sg_host)),
              "hq_host_pipeline_submit")

    def wait(self) -> None:
        check(_lib.load().hq_host_pipeline_wait(self._handle), "hq_host_pipeline_wait")

    def __call__(self, x_host: torch.Tensor):
        self.submit(x_host)
        self.wait()
        return self.q_host, self.s_host, float(self.sg_host[0])

    def inject_failure(self, step: int) -> None:
        """Test of the failure handling (hq_host_pipeline_inject_failure): the next submit()
        behaves as if the CUDA runtime refused its step ``step`` (0 input copy, 1 pass 1, 2 pass 2,
        3 output transfer); nothing on the device fails."""
        check(_lib.load().hq_host_pipeline_inject_failure(self._handle, step),
              "hq_host_pipeline_inject_failure")

    def close(self) -> None:
        if getattr(self, "_handle", None):
            check(_lib.load().hq_host_pipeline_destroy(self._handle), "hq_host_pipeline_destroy")
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
