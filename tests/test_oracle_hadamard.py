"""Pins of the oracle's rotation.

The rotation is defined on "A Fused Hadamard + NVFP4 Quantization Kernel in Triton",
§1 (16x16 Sylvester-Hadamard scaled by 1/4, H.H^T = I) and §2 (hadamard16: H <- [[H, H],
[H, -H]] four times, then / 4).  The 256-point rotation is Sylvester H256 = H16 (x) H16
scaled by 1/16.  These tests tie the oracle's butterfly to scipy's Sylvester construction
(a library routine), to orthonormality, and to the one-hot closed form.
"""
import numpy as np
import pytest
import scipy.linalg

from oracle import rotate, rot_amax


@pytest.mark.parametrize("G", [16, 256])
def test_one_hot_rows_are_scaled_sylvester(oracle_lib, G):
    # e_k . H / sqrt(G) is row k of H / sqrt(G); every entry is +-1/sqrt(G), exact in fp32.
    R = rotate(np.eye(G, dtype=np.float32), G)
    H = scipy.linalg.hadamard(G).astype(np.float64) / np.sqrt(G)
    assert np.array_equal(R.astype(np.float64), H)


@pytest.mark.parametrize("G", [16, 256])
def test_rotation_is_orthonormal_and_symmetric(oracle_lib, G):
    R = rotate(np.eye(G, dtype=np.float32), G).astype(np.float64)
    assert np.array_equal(R @ R.T, np.eye(G))
    assert np.array_equal(R, R.T)


@pytest.mark.parametrize("G", [16, 256])
def test_sign_pattern_is_popcount(oracle_lib, G):
    # Sylvester H[i][j] = (-1)^popcount(i & j)
    R = rotate(np.eye(G, dtype=np.float32), G)
    i = np.arange(G)[:, None]
    j = np.arange(G)[None, :]
    pc = np.vectorize(lambda v: bin(v).count("1"))(i & j)
    assert np.array_equal(np.sign(R), np.where(pc % 2 == 0, 1.0, -1.0))


@pytest.mark.parametrize("G", [16, 256])
def test_butterfly_matches_dense_product(oracle_lib, G):
    rng = np.random.default_rng(123)
    x = rng.standard_normal((64, 4 * G)).astype(np.float32)
    x[:, 5] *= 300.0
    y = rotate(x, G).astype(np.float64)
    H = scipy.linalg.hadamard(G).astype(np.float64) / np.sqrt(G)
    ref = (x.astype(np.float64).reshape(-1, G) @ H).reshape(x.shape)
    # fp32 butterfly vs fp64 dense product: error bounded by a few ulps of the group norm
    norms = np.linalg.norm(x.astype(np.float64).reshape(-1, G), axis=1).repeat(G).reshape(x.shape)
    assert np.max(np.abs(y - ref) / norms) < 1e-6


def test_rotation_inverts_itself(oracle_lib):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((8, 512)).astype(np.float32)
    for G in (16, 256):
        back = rotate(rotate(x, G), G)
        assert np.max(np.abs(back - x)) < 1e-5 * np.max(np.abs(x))


def test_group256_is_kron_of_group16(oracle_lib):
    R16 = rotate(np.eye(16, dtype=np.float32), 16).astype(np.float64)
    R256 = rotate(np.eye(256, dtype=np.float32), 256).astype(np.float64)
    assert np.array_equal(R256, np.kron(R16, R16))


def test_rot_amax_matches_rotated_max(oracle_lib):
    rng = np.random.default_rng(11)
    x = rng.standard_normal((37, 512)).astype(np.float32)
    for G in (0, 16, 256):
        amax, y = rot_amax(x, G, want_y=True, nthreads=3)
        ref = x if G == 0 else rotate(x, G)
        assert np.array_equal(y, ref)
        assert amax == np.max(np.abs(ref))


def test_rot_amax_surfaces_nonfinite(oracle_lib):
    x = np.ones((4, 32), np.float32)
    x[2, 5] = np.inf
    assert np.isinf(rot_amax(x, 0)[0])
    x[1, 1] = np.nan
    assert np.isnan(rot_amax(x, 0)[0])
    assert np.isnan(rot_amax(x, 16)[0])
