"""Seeded synthetic activations and the named workloads.

This module only draws inputs: it holds none of the rotation or quantization
arithmetic, so the CUDA path and the CPU oracle can both consume its bytes.

Recipe (the same for every workload):

* ``root = numpy.random.SeedSequence(seed)``; ``pick, *rows = root.spawn(1 + n_chunks)``
  where the M rows are cut into chunks of ``ROW_CHUNK`` rows.
* Each row chunk ``i`` is drawn by ``Generator(PCG64(rows[i]))``: N(0,1) in fp32
  (``standard_normal(dtype=float32)``) or Student-t with ``df`` degrees of freedom
  (``standard_t``, fp64) times ``t_scale``, cast to fp32.  Chunks are drawn by a
  thread pool; the values do not depend on the thread count.
* Outlier channels: ``Generator(PCG64(pick)).choice(K, n, replace=False)`` with
  ``n = round(frac * K)`` (or an explicit list), multiplied in fp32 by ``factor``.
* Zero rows (if any) are set to +0.0.
* bf16 workloads are the fp32 tensor cast by ``torch`` (round to nearest even).

The shapes and value patterns follow the activation tensors of the
"A Fused Hadamard + NVFP4 Quantization Kernel in Triton" page (§3 test tensor:
N(0,1) with a few channels scaled up; §5 error study: Gaussian, outlier
channels, Student-t with 3 degrees of freedom) at LLM layer sizes.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

ROW_CHUNK = 256


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    dtype: str            # "f32" or "bf16"
    seed: int
    dist: str             # "normal" or "t"
    groups: tuple         # rotation groups exercised: 0 (off), 16, 256
    outlier_frac: float = 0.0
    outlier_cols: tuple = ()
    outlier_factor: float = 1.0
    t_df: float = 3.0
    t_scale: float = 1.0
    zero_rows: int = 0    # rows 0 .. zero_rows-1 are all zero
    roundtrip: bool = False

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def numel(self) -> int:
        return self.M * self.K

    def bytes_in(self) -> int:
        return self.numel * self.elem_bytes

    def bytes_out(self) -> int:
        # packed codes [M, K/2] + E4M3 scales [M, K/16]
        return self.numel // 2 + self.numel // 16

    def describe(self) -> str:
        dist = "N(0,1)" if self.dist == "normal" else f"t(df={self.t_df:g})*{self.t_scale:g}"
        parts = [f"x {self.dtype} [{self.M},{self.K}]", f"seed {self.seed}", dist]
        if self.outlier_cols:
            parts.append(f"channels {','.join(map(str, self.outlier_cols))} x{self.outlier_factor:g}")
        elif self.outlier_frac:
            parts.append(f"{self.outlier_frac * 100:g}% outlier channels x{self.outlier_factor:g}")
        if self.zero_rows:
            parts.append(f"zero rows 0..{self.zero_rows - 1}")
        parts.append("group " + "/".join("off" if g == 0 else str(g) for g in self.groups))
        return ", ".join(parts)


WORKLOADS = {
    "tiny_f32_128x256": Workload("tiny_f32_128x256", 128, 256, "f32", 0, "normal", (16,),
                                 outlier_cols=(3, 77), outlier_factor=40.0, roundtrip=True),
    "bf16_4096x4096": Workload("bf16_4096x4096", 4096, 4096, "bf16", 1, "normal", (16, 0),
                               outlier_frac=0.01, outlier_factor=50.0),
    "bf16_16384x8192_t3": Workload("bf16_16384x8192_t3", 16384, 8192, "bf16", 2, "t", (16,),
                                   t_df=3.0, t_scale=0.5, zero_rows=16),
    "bf16_32768x28672": Workload("bf16_32768x28672", 32768, 28672, "bf16", 3, "normal", (16,),
                                 outlier_frac=0.005, outlier_factor=100.0),
    "bf16_8192x16384_g256": Workload("bf16_8192x16384_g256", 8192, 16384, "bf16", 4, "normal", (256,),
                                     outlier_frac=0.01, outlier_factor=50.0, roundtrip=True),
}

# The order the workloads are listed in (smallest correctness case first).
WORKLOAD_ORDER = ["tiny_f32_128x256", "bf16_4096x4096", "bf16_16384x8192_t3",
                  "bf16_32768x28672", "bf16_8192x16384_g256"]


def outlier_channels(w: Workload) -> np.ndarray:
    if w.outlier_cols:
        return np.array(w.outlier_cols, dtype=np.int64)
    n = int(round(w.outlier_frac * w.K))
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    pick = np.random.SeedSequence(w.seed).spawn(1 + _n_chunks(w.M))[0]
    return np.sort(np.random.Generator(np.random.PCG64(pick)).choice(w.K, n, replace=False))


def _n_chunks(M: int) -> int:
    return max(1, (M + ROW_CHUNK - 1) // ROW_CHUNK)


def generate_f32(w: Workload, rows: slice | None = None, threads: int | None = None) -> np.ndarray:
    """The fp32 activations of ``w`` (before any bf16 cast), optionally only a row range.

    A row range is drawn chunk by chunk from the same streams, so it equals the
    corresponding rows of the full tensor.
    """
    r0, r1 = (0, w.M) if rows is None else (rows.start or 0, w.M if rows.stop is None else rows.stop)
    if not (0 <= r0 <= r1 <= w.M):
        raise ValueError("row range out of bounds")
    kids = np.random.SeedSequence(w.seed).spawn(1 + _n_chunks(w.M))[1:]
    out = np.empty((r1 - r0, w.K), np.float32)
    c0, c1 = r0 // ROW_CHUNK, (r1 + ROW_CHUNK - 1) // ROW_CHUNK

    def draw(ci: int) -> None:
        g = np.random.Generator(np.random.PCG64(kids[ci]))
        lo, hi = ci * ROW_CHUNK, min(w.M, (ci + 1) * ROW_CHUNK)
        if w.dist == "normal":
            block = g.standard_normal((hi - lo, w.K), dtype=np.float32)
        elif w.dist == "t":
            block = (g.standard_t(w.t_df, size=(hi - lo, w.K)) * w.t_scale).astype(np.float32)
        else:
            raise ValueError(w.dist)
        a, b = max(lo, r0), min(hi, r1)
        out[a - r0:b - r0] = block[a - lo:b - lo]

    n_threads = threads or min(32, os.cpu_count() or 1)
    if c1 - c0 <= 1 or n_threads <= 1:
        for ci in range(c0, c1):
            draw(ci)
    else:
        with ThreadPoolExecutor(n_threads) as ex:
            list(ex.map(draw, range(c0, c1)))
    cols = outlier_channels(w)
    if cols.size:
        out[:, cols] *= np.float32(w.outlier_factor)
    if w.zero_rows and r0 < w.zero_rows:
        out[: min(w.zero_rows, r1) - r0] = 0.0
    return out


def generate(w: Workload, rows: slice | None = None, threads: int | None = None) -> torch.Tensor:
    """The input tensor of ``w`` on the host: torch float32 or bfloat16, contiguous."""
    x = torch.from_numpy(generate_f32(w, rows, threads))
    return x if w.dtype == "f32" else x.to(torch.bfloat16)


def as_oracle_array(x: torch.Tensor) -> np.ndarray:
    """Host tensor -> numpy view the oracle takes (float32, or uint16 bf16 bit patterns)."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.float32:
        return x.numpy()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(f"unsupported dtype {x.dtype}")
