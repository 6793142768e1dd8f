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


def torch_blocked_helpers():
    """PyTorch's own statement of the layout, as Python source: ``to_blocked`` and
    ``from_blocked`` in torch/testing/_internal/common_quantized.py, the helpers PyTorch's tests
    use to feed block scales to ``torch._scaled_mm`` (their comments cite cuBLAS's "1D block
    scaling factors layout").  ``to_blocked`` builds the layout with reshapes and a transpose;
    ``from_blocked`` reads it back with the per-element offset formula.  The module itself
    imports test-only packages, so the two functions (and their ``ceil_div``) are taken from its
    source with ``ast`` and run on their own."""
    import ast
    import importlib.util

    import torch

    spec = importlib.util.find_spec("torch.testing._internal.common_quantized")
    if spec is None or spec.origin is None:
        pytest.skip("this torch has no common_quantized.py")
    tree = ast.parse(open(spec.origin).read())
    wanted = {"ceil_div", "to_blocked", "from_blocked"}
    funcs = [n for n in tree.body if isinstance(n, ast.FunctionDef) and n.name in wanted]
    if {f.name for f in funcs} != wanted:
        pytest.skip("this torch's common_quantized.py lacks to_blocked / from_blocked")
    ns = {"torch": torch}
    exec(compile(ast.Module(body=funcs, type_ignores=[]), spec.origin, "exec"), ns)
    return ns["to_blocked"], ns["from_blocked"]


@pytest.mark.parametrize("M,C0", [(1, 1), (31, 3), (128, 4), (129, 5), (200, 6), (256, 8), (300, 17)])
def test_layout_equals_pytorchs_blocked_scale_helpers(M, C0):
    """The oracle's swizzle against an independent statement of the same layout.  Distinct byte
    labels catch a transposed pair of in-tile terms ((r % 32) * 16 + (r / 32) * 4 swapped), a
    wrong tile order or wrong padding, which the bijection test above cannot."""
    import torch

    to_blocked, from_blocked = torch_blocked_helpers()
    rng = np.random.default_rng(M * 7 + C0)
    s = rng.integers(0, 256, (M, C0), dtype=np.uint8)
    ours = swizzle_scales(s)
    theirs = to_blocked(torch.from_numpy(s)).numpy()
    assert theirs.dtype == np.uint8 and theirs.size == ours.size
    assert np.array_equal(ours, theirs)
    # from_blocked takes the [M, K] data tensor only for its shape (K = 16 * C0 for NVFP4)
    data = torch.empty((M, 16 * C0), dtype=torch.uint8)
    back = from_blocked(data, torch.from_numpy(ours), 16).numpy()
    assert np.array_equal(back, s)
