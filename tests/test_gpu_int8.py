"""INT8 per-token rotate-quant (hq_rotate_quant_int8) against the oracle, bit-exact.

"hyperflow_h3_flash_int8.py" (HyperFlow): regular_hadamard, hadamard_factors,
rotate_quant_kernel, rotate_quant.  Groups 4, 16, 64, 256 and 1024 (the page's group sizes:
powers of 4).  Shapes cover one and several warp tiles per row (2048 channels each), ragged last
tiles, 1 to 16 rows per CTA step, rows longer than tensor memory holds (32768 < K <= 120832:
parked in tensor and shared memory; longer: each row read twice), both input types, strided
rows, zero rows (the 1e-12 floor) and extreme magnitudes.
"""
import numpy as np
import pytest
import torch

import hadamard_rotation_gb300 as hq
import oracle
from hadamard_rotation_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from hadamard_rotation_gb300 import build

    build.build()
    oracle.build()
    hq.load()


def rand_input(M, K, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(scale)
    if K >= 64:
        x[:, rng.choice(K, max(1, K // 100), replace=False)] *= 40.0
    if M > 2:
        x[1] = 0.0
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def check(x_host, group, x_dev=None):
    x = x_dev if x_dev is not None else x_host.cuda()
    q, s = hq.hq_rotate_quant_int8(x, group)
    torch.cuda.synchronize()
    oq, os_ = oracle.rotate_quant_int8(synth.as_oracle_array(x_host), group)
    gs = s.cpu().numpy()
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), "scales differ"
    gq = q.cpu().numpy()
    if not np.array_equal(gq, oq):
        bad = np.argwhere(gq != oq)
        raise AssertionError(f"{len(bad)} codes differ, first {bad[:5].tolist()}")


SHAPES = [(1, 16, 16), (3, 48, 16), (17, 64, 64), (5, 256, 256), (33, 2048, 16), (9, 2304, 256),
          (100, 4096, 64), (7, 32768, 256), (1000, 1024, 16), (301, 3072, 64), (64, 6144, 256),
          (40, 30720, 16), (11, 2048 + 192, 64),
          # group 4 (one digit), group 1024 (five digits, two of them across lanes)
          (2, 16, 4), (37, 2064, 4), (5, 1024, 1024), (13, 3072, 1024), (8, 32768, 1024),
          # rows longer than tensor memory holds, parked in tensor and shared memory: 17 warp
          # tiles, a ragged 19th, 32, a ragged 49th, 59 (the most parked on chip)
          (3, 34816, 16), (5, 36864 + 1024, 1024), (4, 65536, 256), (2, 98304 + 16, 4),
          (3, 65536, 64), (3, 120832, 16),
          # 2 or 3 such rows per CTA step (T <= 24): a partial last block, more blocks than SMs
          (301, 36864, 256), (500, 40960, 16), (7, 47104 + 64, 64),
          # longer still, each row read twice: a ragged 60th tile, 60 and 64 tiles
          (2, 120832 + 16, 16), (2, 122880, 256), (2, 131072, 1024), (2, 122880 + 192, 64)]


@pytest.mark.parametrize("M,K,group", SHAPES)
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_int8_parity(M, K, group, dtype):
    check(rand_input(M, K, dtype, seed=M + K + group), group)


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
def test_int8_strided_rows(group):
    big = rand_input(300, 4096 + 512, torch.bfloat16, seed=4)
    check(big[:, :4096].contiguous(), group, x_dev=big.cuda()[:, :4096])


@pytest.mark.parametrize("group", [16, 1024])
def test_int8_long_rows_strided_and_many(group):
    """Rows of 65536 channels (parked on chip), strided, more rows than SMs."""
    big = rand_input(400, 65536 + 1024, torch.bfloat16, seed=7)
    check(big[:, :65536].contiguous(), group, x_dev=big.cuda()[:, :65536])


@pytest.mark.parametrize("scale", [1e-30, 1e-14, 1e30])
def test_int8_extreme_magnitudes(scale):
    for group in (4, 16, 64, 256, 1024):
        check(rand_input(50, 1024, torch.float32, seed=9, scale=scale), group)
    check(rand_input(3, 40960, torch.float32, seed=10, scale=scale), 256)   # a long row


def test_int8_llm_sized_workload():
    w = synth.Workload("int8_bf16_8192x8192", 8192, 8192, "bf16", 5, "normal", (256,),
                       outlier_frac=0.01, outlier_factor=50.0)
    x = synth.generate(w)
    for group in (64, 256):
        check(x, group)


def test_int8_empty_and_limits():
    x = torch.empty(0, 256, device="cuda", dtype=torch.bfloat16)
    q, s = hq.hq_rotate_quant_int8(x, 256)
    assert q.numel() == 0
    with pytest.raises(hq.HQError):
        hq.hq_rotate_quant_int8(torch.zeros(2, 1536, device="cuda", dtype=torch.bfloat16), 1024)


def _tie_row(group):
    """One fp32 row of 2 * group channels whose rotated value y satisfies
    RN(y * inv) = k + 1/2 exactly while the exact product y * inv is not k + 1/2:
    rint of the rounded product (the definition) and of an unrounded one (a fused
    multiply-add) differ.  A one-hot value v in a group rotates to +-v / sqrt(G) on
    every channel, exactly, so group 0 fixes the row amax and group 1 carries y."""
    r = np.float32(np.sqrt(group))
    for amax in np.linspace(10.0, 60.0, 2001, dtype=np.float32):
        scale = np.float32(amax / np.float32(127.0))
        inv = np.float32(np.float32(1.0) / scale)
        for k in range(20, 40):
            y = np.float32((k + 0.5) / float(inv))
            for _ in range(32):
                y = np.nextafter(y, np.float32(-np.inf))
            for _ in range(64):
                prod = np.float32(y * inv)
                exact = float(y) * float(inv)  # 24 x 24 bits: exact in float64
                if float(prod) == k + 0.5 and np.rint(exact) != np.rint(prod):
                    row = np.zeros(2 * group, np.float32)
                    row[0] = amax * r
                    row[group] = y * r
                    assert row[0] / r == amax and row[group] / r == y
                    return row
                y = np.nextafter(y, np.float32(np.inf))
    raise AssertionError("no tie case found")


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
def test_int8_rint_of_rounded_product(group):
    """q = rint(RN(y * (1/scale))): the product is rounded before rint."""
    row = _tie_row(group)
    row = np.concatenate([row, np.zeros(-row.size % 16, np.float32)])  # whole 16-channel blocks
    x = torch.from_numpy(np.tile(row, (4, 1)))
    check(x, group)
