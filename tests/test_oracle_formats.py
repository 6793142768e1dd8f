"""Exhaustive pins of the oracle's two roundings: fp32 -> E2M1 code and fp32 -> E4M3 scale.

Sources: "A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 table (E2M1 grid
{0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3 block scale), §2 (_e2m1_code: midpoints, ties to the even
code; _round_e4m3: minimum normal 2^-6, 3 mantissa bits, clamp 448), §3 (the
round-to-nearest-even float8_e4m3fn cast), §4 (printed cast examples).
The checks use rules that are independent of the oracle's implementation: the grid and the
tie rule in bit space, a brute-force nearest search in float64, and torch's float8_e4m3fn cast.
"""
import numpy as np
import pytest
import torch

from conftest import load_golden
from oracle import e2m1_codes, e2m1_codes_bits, e4m3_codes, e4m3_codes_bits, e4m3_values

FMT = load_golden("p1_format.txt")
GRID = np.array([float(v) for v in FMT["e2m1_grid"]])
CHUNK = 1 << 27


def f32_bits(v: float) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


# ---------------------------------------------------------------- E2M1 -----------------

def expected_e2m1_transitions():
    """Bit patterns where the magnitude code steps k -> k+1, from the grid and the tie rule.

    Between grid[k] and grid[k+1] the midpoint m is exactly representable.  A value equal
    to m goes to the even code: if k is even the code stays k at m (step at bits(m) + 1),
    otherwise it becomes k+1 at m (step at bits(m)).
    """
    steps = []
    for k in range(7):
        m = (GRID[k] + GRID[k + 1]) / 2.0
        steps.append(f32_bits(m) + (1 if k % 2 == 0 else 0))
    return steps


def test_e2m1_midpoints_match_page(oracle_lib):
    mids = [float(v) for v in FMT["e2m1_midpoints"]]
    assert mids == [(GRID[k] + GRID[k + 1]) / 2 for k in range(7)]


def test_e2m1_exhaustive_nonnegative(oracle_lib):
    """All non-negative fp32 patterns 0 .. +inf: monotone, 7 steps exactly where expected."""
    last = 0x7F800000  # +inf, saturates like any finite value above 5
    found = []
    prev = None
    for first in range(0, last + 1, CHUNK):
        n = min(CHUNK, last + 1 - first)
        c = e2m1_codes_bits(first, n)
        assert c.max() <= 7
        if prev is not None and c[0] != prev:
            assert c[0] == prev + 1
            found.append(first)
        d = np.diff(c.astype(np.int16))
        assert d.min() >= 0 and d.max() <= 1
        found.extend((first + 1 + np.flatnonzero(d)).tolist())
        prev = int(c[-1])
    assert found == expected_e2m1_transitions()
    assert prev == 7


def test_e2m1_exhaustive_sign(oracle_lib):
    """code(-v) == code(v) | 8 for every non-negative pattern v (including -0.0 -> 8)."""
    last = 0x7F800000
    for first in range(0, last + 1, CHUNK):
        n = min(CHUNK, last + 1 - first)
        pos = e2m1_codes_bits(first, n)
        neg = e2m1_codes_bits(0x80000000 + first, n)
        assert np.array_equal(neg, pos | 8)


def brute_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest grid value in float64, ties to the even code, saturating at 6; sign bit copied."""
    a = np.minimum(np.abs(v.astype(np.float64)), 6.0)
    dist = np.abs(a[:, None] - GRID[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(8)[None, :] % 2 == 0)
    code = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    return (code | (np.signbit(v) * 8)).astype(np.uint8)


def test_e2m1_brute_force_near_every_decision_point(oracle_lib):
    vals = []
    for p in list(GRID) + [(GRID[k] + GRID[k + 1]) / 2 for k in range(7)] + [6.5, 1e30]:
        b = f32_bits(p)
        vals.append(np.arange(max(0, b - 2000), b + 2000, dtype=np.uint32).view(np.float32))
    rng = np.random.default_rng(5)
    vals.append((rng.random(2_000_000) * 8).astype(np.float32))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    assert np.array_equal(e2m1_codes(v), brute_e2m1(v))


def test_e2m1_all_codes_round_trip(oracle_lib):
    vals = np.concatenate([GRID, -GRID]).astype(np.float32)
    codes = e2m1_codes(vals)
    assert codes.tolist() == list(range(8)) + list(range(8, 16))


# ---------------------------------------------------------------- E4M3 -----------------

def e4m3_table():
    """The 127 non-negative finite E4M3 values from the bit layout (bias 7, 3 mantissa bits)."""
    codes = np.arange(127)
    ef, m = codes >> 3, codes & 7
    return np.where(ef == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (ef - 7))


def brute_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest of the 127 finite values in float64, ties to the even mantissa, clamp 448."""
    table = e4m3_table()
    a = np.minimum(v.astype(np.float64), 448.0)
    dist = np.abs(a[:, None] - table[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(127)[None, :] % 2 == 0)
    return np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1)).astype(np.uint8)


def test_e4m3_format_constants(oracle_lib):
    t = e4m3_table()
    assert t.max() == float(FMT["e4m3_max"][0])
    assert t[8] == float(FMT["e4m3_min_normal"][0])       # exponent field 1, mantissa 0
    assert e4m3_values(np.arange(127, dtype=np.uint8)).astype(np.float64).tolist() == t.tolist()


def test_e4m3_decode_matches_torch(oracle_lib):
    codes = np.arange(127, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(e4m3_values(codes), ref)


def test_e4m3_page_examples(oracle_lib):
    g = load_golden("p1_cast_repro.txt")
    x = np.array([float(v) for v in g["input"]], np.float32)
    want = [float(v) for v in g["rtne"]]
    assert e4m3_values(e4m3_codes(x)).tolist() == want


def test_e4m3_special_values(oracle_lib):
    cases = {448.0: 448.0, 460.0: 448.0, 1e30: 448.0, float("inf"): 448.0,
             2.0 ** -6: 2.0 ** -6, 2.0 ** -9: 2.0 ** -9, 2.0 ** -10: 0.0,
             3 * 2.0 ** -10: 2.0 ** -8, 0.0: 0.0, 1e-45: 0.0}
    x = np.array(list(cases), np.float32)
    assert e4m3_values(e4m3_codes(x)).tolist() == list(cases.values())


def test_e4m3_exhaustive_vs_torch_cast(oracle_lib):
    """Every fp32 in [2^-11, 448]: the oracle equals torch's RNE float8_e4m3fn cast."""
    lo, hi = f32_bits(2.0 ** -11), f32_bits(448.0)
    for first in range(lo, hi + 1, CHUNK):
        n = min(CHUNK, hi + 1 - first)
        v = np.arange(first, first + n, dtype=np.uint32).view(np.float32)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(e4m3_codes_bits(first, n), ref)


def test_e4m3_exhaustive_below_half_min_subnormal(oracle_lib):
    """Every fp32 in [0, 2^-11) rounds to 0 (below half of the smallest subnormal 2^-9)."""
    hi = f32_bits(2.0 ** -11)
    for first in range(0, hi, CHUNK):
        n = min(CHUNK, hi - first)
        assert not e4m3_codes_bits(first, n).any()


def test_e4m3_saturates_above_448(oracle_lib):
    lo = f32_bits(448.0)
    c = e4m3_codes_bits(lo, f32_bits(2.0 ** 20) - lo)       # exhaustive [448, 2^20)
    assert (c == 0x7E).all()
    rest = np.arange(f32_bits(2.0 ** 20), 0x7F800001, 4099, dtype=np.uint32).view(np.float32)
    assert (e4m3_codes(rest) == 0x7E).all()


def test_e4m3_brute_force_sample(oracle_lib):
    rng = np.random.default_rng(9)
    v = np.concatenate([
        (rng.random(300_000) * 500).astype(np.float32),
        np.exp2(rng.uniform(-14, 9, 300_000)).astype(np.float32),
        # every midpoint between neighbouring values, and one ulp either side
        np.repeat((e4m3_table()[:-1] + e4m3_table()[1:]) / 2, 3).astype(np.float32),
    ])
    mids = (e4m3_table()[:-1] + e4m3_table()[1:]) / 2
    m32 = mids.astype(np.float32)
    v = np.concatenate([v, np.nextafter(m32, np.float32(0)), np.nextafter(m32, np.float32(1e9))])
    assert np.array_equal(e4m3_codes(v), brute_e4m3(v))
