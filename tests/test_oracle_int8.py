"""Pins of the oracle's INT8 per-token rotate-quant ("hyperflow_h3_flash_int8.py", HyperFlow:
regular_hadamard, hadamard_factors, rotate_quant_kernel).

The regular Hadamard is tied to the h4 matrix the page prints (tests/golden), to the properties
its docstring states (orthonormal, symmetric, rows summing to one), to the page's factoring
R_256 = kron(R_16, R_16) and to an fp64 dense product.  The quantizer is tied to a closed form
(one non-zero channel gives +-127 with the matrix's signs), the zero-row floor, the rounding
error bound and the nearest-integer property in float64.
"""
import numpy as np
import pytest

from conftest import load_golden
from oracle import int8_rotate, rotate_quant_int8

G = load_golden("p3_regular_hadamard.txt")
H4 = np.array([[float(v) for v in G[f"h4_row{i}"]] for i in range(4)]) / float(G["h4_divisor"][0])


def kron_power(n):
    r = np.ones((1, 1))
    while r.shape[0] < n:
        r = np.kron(r, H4)
    return r


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
def test_rotation_is_the_pages_kronecker_power(oracle_lib, group):
    R = int8_rotate(np.eye(group, dtype=np.float32), group).astype(np.float64)
    assert np.array_equal(R, kron_power(group))


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
def test_rotation_properties_from_the_docstring(oracle_lib, group):
    R = int8_rotate(np.eye(group, dtype=np.float32), group).astype(np.float64)
    assert np.array_equal(R @ R.T, np.eye(group))       # orthonormal
    assert np.array_equal(R, R.T)                       # symmetric
    assert np.array_equal(R.sum(axis=1), np.ones(group))  # rows sum to one


def test_factoring_of_1024_as_16_by_64(oracle_lib):
    # HyperFlow's hadamard_factors computes a group of 1024 as factors 16 and 64: the
    # Kronecker product of the two smaller rotations is the group-1024 rotation.
    R = int8_rotate(np.eye(1024, dtype=np.float32), 1024).astype(np.float64)
    R16 = int8_rotate(np.eye(16, dtype=np.float32), 16).astype(np.float64)
    R64 = int8_rotate(np.eye(64, dtype=np.float32), 64).astype(np.float64)
    assert np.array_equal(R, np.kron(R16, R64)) and np.array_equal(R, np.kron(R64, R16))


def test_factoring_of_256(oracle_lib):
    ga, gb = (int(v) for v in G["factors_256"])
    R = int8_rotate(np.eye(256, dtype=np.float32), 256).astype(np.float64)
    Ra = int8_rotate(np.eye(ga, dtype=np.float32), ga).astype(np.float64)
    Rb = int8_rotate(np.eye(gb, dtype=np.float32), gb).astype(np.float64)
    assert np.array_equal(R, np.kron(Ra, Rb))


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
def test_fp32_evaluation_matches_dense_product(oracle_lib, group):
    rng = np.random.default_rng(group)
    x = rng.standard_normal((32, 4 * group)).astype(np.float32)
    x[:, 3] *= 500.0
    y = int8_rotate(x, group).astype(np.float64)
    ref = (x.astype(np.float64).reshape(-1, group) @ kron_power(group)).reshape(x.shape)
    norms = np.linalg.norm(x.astype(np.float64).reshape(-1, group), axis=1).repeat(group).reshape(x.shape)
    assert np.max(np.abs(y - ref) / norms) < 1e-6


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
@pytest.mark.parametrize("c", [1.0, -7.5, 3e-8, 2e30])
def test_single_channel_closed_form(oracle_lib, group, c):
    K = 2 * group
    for p in (0, 1, group - 1):
        x = np.zeros((2, K), np.float32)
        x[1, group + p] = c
        q, s = rotate_quant_int8(x, group)
        assert not q[0].any() and not q[1, :group].any()
        want = np.where(np.sign(kron_power(group)[p]) * np.sign(c) > 0, 127, -127)
        assert q[1, group:].tolist() == want.tolist()


def test_zero_row_uses_the_floor(oracle_lib):
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = 1e-20
    q, s = rotate_quant_int8(x, 16)
    floor = np.float32(float(G["scale_floor"][0])) / np.float32(127.0)
    assert s[0] == floor and s[2] == floor and not q[0].any()
    assert s[1] == floor       # amax 1e-20 / 2 is below 1e-12


@pytest.mark.parametrize("group", [4, 16, 64, 256, 1024])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_codes_are_nearest_integers_within_the_bound(oracle_lib, group, dtype):
    import torch

    rng = np.random.default_rng(5 + group)
    x = rng.standard_normal((64, 1024)).astype(np.float32)
    x[:, [7, 300]] *= 60.0
    x[10] = 0.0
    xin = x if dtype == "f32" else torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xf = x if dtype == "f32" else torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    q, s = rotate_quant_int8(xin, group)
    y = int8_rotate(xf, group)
    amax = np.abs(y).max(axis=1)
    assert np.array_equal(s, np.maximum(amax, np.float32(1e-12)) / np.float32(127.0))
    inv = (np.float32(1.0) / s)[:, None]
    t = (y * inv).astype(np.float64)                 # the fp32 product, exactly
    qd = q.astype(np.float64)
    assert np.all(np.abs(t - qd) <= 0.5)             # nearest integer
    ties = np.abs(t - np.trunc(t)) == 0.5
    assert np.all(qd[ties] % 2 == 0)                 # ties to even
    assert np.abs(q.astype(int)).max() <= int(G["int8_max"][0])
    nz = amax > 1e-12
    assert np.all(np.abs(q[nz].astype(int)).max(axis=1) == 127)   # the amax element maps to 127
    # |q s - y| <= s (|q - y inv| + |y| |inv - 1/s|) <= s (0.5 + 127 * 2^-24 * (1 + tiny))
    err = np.abs(qd * s[:, None].astype(np.float64) - y.astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 2.0 ** -16))


def test_multiply_by_reciprocal_vs_divide_reading(oracle_lib):
    """The page's kernel multiplies by inv = 1 / scale; its torch fallback divides by scale.
    The oracle follows the kernel.  The two differ on a small share of values."""
    rng = np.random.default_rng(1)
    y = (rng.standard_normal(1_000_000) * 30).astype(np.float32)
    scale = np.float32(np.abs(y).max()) / np.float32(127.0)
    a = np.rint(y * (np.float32(1.0) / scale))
    b = np.rint(y / scale)
    frac = np.mean(a != b)
    assert frac < 0.01
