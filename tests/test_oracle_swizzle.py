"""Structure of the oracle's swizzled block-scale layout (swizzle_scales).

"A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §6 "From interpreter to hardware"
(Layout): NVFP4 GEMMs take the block scales in a swizzled tiled layout that the page does not
spell out; the reading is cuBLASLt's layout for 16-element block scales.  What the layout
means is pinned on the GPU, where the library's swizzled scales drive cuBLASLt's NVFP4 GEMM
(tests/test_gpu_swizzle.py).  Here: it is a bijection from the scale matrix onto the padded
buffer, each 128 x 4 tile of the matrix fills 512 consecutive bytes, and padding stays zero.
"""
import numpy as np
import pytest

from oracle import swizzle_scales, unswizzle_scales


def padded(M, C0):
    return (-(-M // 128) * 128) * (-(-C0 // 4) * 4)


@pytest.mark.parametrize("M,C0", [(1, 1), (128, 4), (129, 5), (200, 6), (256, 8), (300, 17)])
def test_bijection_and_padding(M, C0):
    rng = np.random.default_rng(M * 31 + C0)
    s = rng.integers(1, 256, (M, C0), dtype=np.uint8)
    buf = swizzle_scales(s)
    assert buf.size == padded(M, C0)
    assert np.array_equal(unswizzle_scales(buf, M, C0), s)
    # every matrix entry has its own byte: tag entries with distinct labels
    lab = np.arange(M * C0).reshape(M, C0)
    hits = np.zeros(buf.size, np.int64)
    for v in range(3):  # three bytes of the label, one pass each
        b = swizzle_scales(((lab >> (8 * v)) & 0xFF).astype(np.uint8)).astype(np.int64)
        hits |= b << (8 * v)
    nz = np.zeros(buf.size, bool)
    nz[swizzle_scales(np.ones((M, C0), np.uint8)).astype(bool)] = True
    assert nz.sum() == M * C0
    assert sorted(hits[nz].tolist()) == list(range(M * C0))
    assert not buf[~nz].any()                   # padding is zero


def test_tiles_are_contiguous():
    M, C0 = 256, 8
    tile_of = np.zeros((M, C0), np.uint8)
    for r in range(M):
        for c in range(C0):
            tile_of[r, c] = 1 + (r // 128) * 2 + c // 4   # tiles labelled 1..4, row-major
    buf = swizzle_scales(tile_of)
    for t in range(4):
        assert np.all(buf[t * 512:(t + 1) * 512] == t + 1)
