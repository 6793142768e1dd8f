"""GPU vs CPU oracle, through the C ABI.  Codes, scales, amax, s_global and dequantized
values must be bit-exact; the exposed rotated tensor y must be too (the contract allows 1e-6
relative; the butterfly order is the same, so it is exact).

Workloads are the five named activation tensors (synth.WORKLOADS) at full size, run with the
same entry points and launch configuration as bench.py, plus edge cases: a single block, ragged
tiles, strided rows, all-zero and underflowing tensors, extreme magnitudes (the kernel's exact
slow path), non-finite input, another stream, and tiling invariance.
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


def f32_bits(a) -> np.ndarray:
    return np.asarray(a, np.float32).view(np.uint32)


def first_diffs(a: np.ndarray, b: np.ndarray, n=5):
    idx = np.argwhere(a != b)[:n]
    return [(tuple(i), int(a[tuple(i)]), int(b[tuple(i)])) for i in idx]


def assert_bytes_equal(name, gpu: np.ndarray, ref: np.ndarray):
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    if not np.array_equal(gpu, ref):
        bad = int(np.count_nonzero(gpu != ref))
        raise AssertionError(f"{name}: {bad} of {gpu.size} differ; first: {first_diffs(gpu, ref)}")


def gpu_quantize(x_host: torch.Tensor, group: int, want_y=False, stream=None, x_dev=None):
    x = x_dev if x_dev is not None else x_host.cuda()
    y = torch.empty(x.shape, dtype=torch.float32, device=x.device) if want_y else None
    amax = hq.hq_rot_amax(x, group, y=y, stream=stream)
    q, s, sg = hq.hq_rotate_quant_nvfp4(x, group, amax, stream=stream)
    torch.cuda.synchronize()
    out = dict(q=q.cpu().numpy(), s=s.cpu().numpy(), amax=amax.cpu().numpy(), sg=sg.cpu().numpy())
    if want_y:
        out["y"] = y.cpu().numpy()
    out["_dev"] = (q, s, sg)
    return out


def check_against_oracle(x_host: torch.Tensor, group: int, want_y=False, x_dev=None, label=""):
    g = gpu_quantize(x_host, group, want_y=want_y, x_dev=x_dev)
    xo = synth.as_oracle_array(x_host)
    oq, os_, oamax, osg = oracle.quantize(xo, group)
    tag = f"{label} group={group}"
    assert f32_bits(g["amax"])[0] == f32_bits([oamax])[0], (tag, g["amax"], oamax)
    assert f32_bits(g["sg"])[0] == f32_bits([osg])[0], (tag, g["sg"], osg)
    assert_bytes_equal(f"{tag} scales", g["s"], os_)
    assert_bytes_equal(f"{tag} codes", g["q"], oq)
    if want_y:
        _, oy = oracle.rot_amax(xo, group, want_y=True)
        assert_bytes_equal(f"{tag} y", f32_bits(g["y"]), f32_bits(oy))
    return g, (oq, os_, oamax, osg)


# ---------------------------------------------------------------- the named workloads ------

@pytest.mark.parametrize("name", synth.WORKLOAD_ORDER)
def test_workload_parity(name):
    w = synth.WORKLOADS[name]
    x_host = synth.generate(w)
    x_dev = x_host.cuda()
    for group in w.groups:
        g, (oq, os_, oamax, osg) = check_against_oracle(x_host, group, x_dev=x_dev, label=name)
        if w.roundtrip:
            q, s, sg = g["_dev"]
            back = hq.hq_dequant_nvfp4(q, s, sg, group, unrotate=True)
            torch.cuda.synchronize()
            ref = oracle.dequant(oq, os_, osg, group, True)
            assert_bytes_equal(f"{name} dequant", f32_bits(back.cpu().numpy()), f32_bits(ref))
        del g
    if w.zero_rows:
        g = gpu_quantize(x_host, w.groups[0], x_dev=x_dev)
        assert not g["s"][: w.zero_rows].any() and not g["q"][: w.zero_rows].any()


# ---------------------------------------------------------------- shapes and edge cases ----

def rand_input(M, K, dtype, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    if outliers and K >= 16:
        cols = rng.choice(K, max(1, K // 64), replace=False)
        x[:, cols] *= 30.0
    if M > 3:
        x[2] = 0.0
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


SHAPES = [
    (1, 16, 0), (1, 16, 16), (2, 256, 256), (17, 48, 16), (3, 272, 16), (129, 256, 256),
    (5, 768, 256), (1000, 272, 0), (257, 1024, 16), (31, 4096, 256), (4099, 96, 16),
]


@pytest.mark.parametrize("M,K,group", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_shapes_and_ragged_tails(M, K, group, dtype):
    x = rand_input(M, K, dtype, seed=M * 7 + K + group)
    check_against_oracle(x, group, want_y=True, label=f"{M}x{K}")


@pytest.mark.parametrize("group", [16, 256])
def test_first_stage_rounding_cancellation_and_signed_zeros(group):
    """bf16 rows whose adjacent pairs need rounding in the first butterfly stage (exponent gaps
    of 0 to 40 between x[2m] and x[2m + 1], magnitudes 2^-60 to 2^60), exact cancellations,
    signed zeros in every combination and subnormal bf16 values.  The kernels may fold the
    widening of bf16 into that stage; every rotated value must still equal the definition's
    (y compared bit for bit), and so must the amax, scales and codes."""
    rng = np.random.default_rng(4242 + group)
    M, K = 64, 1024
    a = (rng.standard_normal((M, K // 2)) * np.exp2(rng.integers(-60, 60, (M, K // 2)))).astype(np.float32)
    b = a * np.exp2(-rng.integers(0, 40, (M, K // 2))) * rng.choice([-1.0, 1.0], (M, K // 2))
    x = np.empty((M, K), np.float32)
    x[:, 0::2] = a
    x[:, 1::2] = b.astype(np.float32)
    x[0, 1::2] = -x[0, 0::2]                                    # x[2m] + x[2m + 1] = 0
    x[1, 1::2] = x[1, 0::2]                                     # x[2m] - x[2m + 1] = 0
    x[2] = np.where(rng.random(K) < 0.5, np.float32(0.0), np.float32(-0.0))
    x[3] = (rng.integers(-100, 100, K) * 2.0 ** -133).astype(np.float32)  # bf16 subnormals
    x[4, 0::2] = -0.0
    check_against_oracle(torch.from_numpy(x).to(torch.bfloat16), group, want_y=True, label="first stage")


@pytest.mark.parametrize("group", [0, 16, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_strided_rows(group, dtype):
    big = rand_input(300, 1024 + 256, dtype, seed=11)
    x_dev = big.cuda()[:, :1024]
    assert x_dev.stride(0) == 1280
    view_host = big[:, :1024].contiguous()
    check_against_oracle(view_host, group, x_dev=x_dev, label="strided")
    # strided device input, strided host input to the oracle: both agree with contiguous
    g1 = gpu_quantize(view_host, group)
    g2 = gpu_quantize(view_host, group, x_dev=x_dev)
    assert_bytes_equal("strided vs contiguous codes", g2["q"], g1["q"])


@pytest.mark.parametrize("group", [0, 16, 256])
def test_dequant_parity(group):
    x = rand_input(64, 512, torch.float32, seed=5)
    for unrotate in ([False, True] if group else [False]):
        g, (oq, os_, oamax, osg) = check_against_oracle(x, group)
        q, s, sg = g["_dev"]
        back = hq.hq_dequant_nvfp4(q, s, sg, group if group else 16, unrotate=unrotate)
        torch.cuda.synchronize()
        ref = oracle.dequant(oq, os_, osg, group, unrotate)
        assert_bytes_equal(f"dequant g={group} un={unrotate}", f32_bits(back.cpu().numpy()), f32_bits(ref))


@pytest.mark.parametrize("scale_exp", [-140, -125, -100, -60, 60, 100, 110])
@pytest.mark.parametrize("group", [0, 16, 256])
def test_extreme_magnitudes_use_exact_path(scale_exp, group):
    """Tensors scaled far from 1: s_f leaves the fast division domain (or y becomes subnormal),
    so the kernel takes its literal-division path; results must still equal the oracle."""
    x = rand_input(40, 512, torch.float32, seed=abs(scale_exp) + group)
    x = (x.double() * 2.0 ** scale_exp).float()
    x[7, :16] = torch.tensor(np.float32(2.0 ** scale_exp) * np.arange(16, dtype=np.float32) * 1e-3)
    check_against_oracle(x, group, want_y=True, label=f"2^{scale_exp}")


def test_mixed_magnitudes_in_one_tensor():
    """Blocks of very different size in one tensor: tiny blocks get zero or subnormal scales."""
    x = rand_input(64, 1024, torch.float32, seed=3)
    x[10:20] *= 1e-30
    x[20:30] *= 1e-38
    x[30, 5] = 3.0e38
    for group in (0, 16, 256):
        check_against_oracle(x, group, label="mixed")


def test_zero_and_underflowing_tensors():
    for x in (torch.zeros(8, 64), torch.full((8, 64), 1e-44), -torch.zeros(8, 64)):
        for group in (0, 16):
            g, _ = check_against_oracle(x, group, label="zero")
            assert g["sg"][0] == 1.0
            assert not g["q"].any() and not g["s"].any()


def test_nonfinite_input_surfaces_in_amax():
    x = torch.ones(64, 256, device="cuda")
    x[33, 7] = float("inf")
    for group in (0, 16, 256):
        assert torch.isinf(hq.hq_rot_amax(x, group)).item()
    x[12, 200] = float("nan")
    for group in (0, 16, 256):
        assert torch.isnan(hq.hq_rot_amax(x, group)).item()


def test_empty_tensor():
    x = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    amax = hq.hq_rot_amax(x, 16)
    q, s, sg = hq.hq_rotate_quant_nvfp4(x, 16, amax)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and q.numel() == 0 and s.numel() == 0


def test_other_stream_and_repeat_calls():
    x_host = rand_input(512, 2048, torch.bfloat16, seed=9)
    ref = gpu_quantize(x_host, 16)
    s = torch.cuda.Stream()
    x = x_host.cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(3):
            amax = hq.hq_rot_amax(x, 16, stream=s)
            q, sc, sg = hq.hq_rotate_quant_nvfp4(x, 16, amax, stream=s)
    s.synchronize()
    assert_bytes_equal("stream codes", q.cpu().numpy(), ref["q"])
    assert_bytes_equal("stream scales", sc.cpu().numpy(), ref["s"])


def test_tiling_invariance():
    """A row's codes do not depend on which tile, warp or CTA handled it: quantizing a slice of
    rows with the full tensor's amax reproduces those rows of the full result."""
    x_host = rand_input(3000, 768, torch.bfloat16, seed=21)
    x = x_host.cuda()
    for group in (0, 16, 256):
        amax = hq.hq_rot_amax(x, group)
        q, s, _ = hq.hq_rotate_quant_nvfp4(x, group, amax)
        for r0, r1 in ((0, 1), (5, 6), (123, 1187), (2999, 3000)):
            qs, ss, _ = hq.hq_rotate_quant_nvfp4(x[r0:r1], group, amax)
            torch.cuda.synchronize()
            assert torch.equal(qs, q[r0:r1]) and torch.equal(ss, s[r0:r1])


def test_host_pipeline_matches_oracle_over_overlapping_submissions():
    """Five submissions in flight through the two-slot host pipeline, each with its own input
    and output buffers; every result must equal the oracle's for its own input."""
    M, K = 1024, 2048
    hqz = hq.HostQuantizer(M, K, torch.bfloat16, 16)
    xs, outs = [], []
    for i in range(5):
        x = rand_input(M, K, torch.bfloat16, seed=100 + i).pin_memory()
        q = torch.empty((M, K // 2), dtype=torch.uint8, pin_memory=True)
        s = torch.empty((M, K // 16), dtype=torch.uint8, pin_memory=True)
        sg = torch.empty(1, dtype=torch.float32, pin_memory=True)
        hqz.submit(x, q, s, sg)
        xs.append(x)
        outs.append((q, s, sg))
    hqz.wait()
    for x, (q, s, sg) in zip(xs, outs):
        oq, os_, oamax, osg = oracle.quantize(synth.as_oracle_array(x), 16)
        assert_bytes_equal("pipeline codes", q.numpy(), oq)
        assert_bytes_equal("pipeline scales", s.numpy(), os_)
        assert np.float32(sg.item()) == osg
    hqz.close()


@pytest.mark.parametrize("pinned_outputs", [True, False])
def test_host_pipeline_output_buffers_of_any_kind(pinned_outputs):
    """Outputs into pinned buffers (stored by the pipeline's copy-out kernel) and into plain
    pageable buffers (stored the same way where the device reaches pageable memory through the
    host page tables, else copied), with odd sizes and offsets: all equal the oracle."""
    M, K = 333, 1040
    hqz = hq.HostQuantizer(M, K, torch.bfloat16, 16)
    x = rand_input(M, K, torch.bfloat16, seed=77).pin_memory()
    # buffers that start 1 byte into a larger allocation: no 16-byte alignment
    qa = torch.empty(M * (K // 2) + 1, dtype=torch.uint8, pin_memory=pinned_outputs)
    sa = torch.empty(M * (K // 16) + 1, dtype=torch.uint8, pin_memory=pinned_outputs)
    q, s = qa[1:].view(M, K // 2), sa[1:].view(M, K // 16)
    sg = torch.empty(1, dtype=torch.float32, pin_memory=pinned_outputs)
    for _ in range(3):
        hqz.submit(x, q, s, sg)
    hqz.wait()
    oq, os_, oamax, osg = oracle.quantize(synth.as_oracle_array(x), 16)
    assert_bytes_equal("pipeline codes", q.numpy(), oq)
    assert_bytes_equal("pipeline scales", s.numpy(), os_)
    assert np.float32(sg.item()) == osg
    hqz.close()


@pytest.mark.parametrize("step", [0, 1, 2, 3])
def test_host_pipeline_refuses_submissions_after_a_partial_failure(step):
    """A submission whose step `step` is refused (injected on the host: the device sees no
    failure) returns HQ_ERR_CUDA.  Once part of it was enqueued (a refused pass 1, pass 2 or
    output transfer), the pipeline refuses every later submission, since the buffer set's
    events may not cover the work in flight; a refused input copy enqueued nothing and leaves it
    usable.  The submissions before the failure still complete and equal the oracle."""
    from hadamard_rotation_gb300._lib import HQ_ERR_CUDA, HQError

    M, K = 256, 1024
    hqz = hq.HostQuantizer(M, K, torch.bfloat16, 16)
    x = rand_input(M, K, torch.bfloat16, seed=31).pin_memory()
    first = [torch.empty((M, K // 2), dtype=torch.uint8, pin_memory=True),
             torch.empty((M, K // 16), dtype=torch.uint8, pin_memory=True),
             torch.empty(1, dtype=torch.float32, pin_memory=True)]
    hqz.submit(x, *first)                       # a good submission before the failure
    hqz.inject_failure(step)
    with pytest.raises(HQError) as err:
        hqz.submit(x)
    assert err.value.status == HQ_ERR_CUDA
    if step == 0:
        hqz.submit(x)                           # nothing was enqueued: still usable
    else:
        with pytest.raises(HQError) as again:
            hqz.submit(x)
        assert again.value.status == HQ_ERR_CUDA
    hqz.wait()
    oq, os_, oamax, osg = oracle.quantize(synth.as_oracle_array(x), 16)
    assert_bytes_equal("codes before the failure", first[0].numpy(), oq)
    assert_bytes_equal("scales before the failure", first[1].numpy(), os_)
    if step == 0:
        assert_bytes_equal("codes after a refused copy", hqz.q_host.numpy(), oq)
    hqz.close()
    assert torch.cuda.synchronize() is None     # the context is still usable


def test_host_quantizer_matches_oracle_on_a_workload():
    w = synth.WORKLOADS["bf16_4096x4096"]
    x_host = synth.generate(w).pin_memory()
    hqz = hq.HostQuantizer(w.M, w.K, torch.bfloat16, 16)
    qh, sh, sg = hqz(x_host)
    oq, os_, oamax, osg = oracle.quantize(synth.as_oracle_array(x_host), 16)
    assert_bytes_equal("host codes", qh.numpy(), oq)
    assert_bytes_equal("host scales", sh.numpy(), os_)
    assert np.float32(sg) == osg
    hqz.close()


@pytest.mark.parametrize("group", [0, 16])
def test_pass1_on_16_byte_aligned_input(group):
    """x whose base is 16- but not 32-byte aligned takes pass 1's TMA path instead of the
    streaming one; both must give the oracle's amax."""
    M, K = 257, 1024
    x_host = rand_input(M, K, torch.bfloat16, seed=77)
    flat = torch.empty(M * K + 8, dtype=torch.bfloat16, device="cuda")
    x_dev = flat[8:].view(M, K)
    x_dev.copy_(x_host)
    assert x_dev.data_ptr() % 32 == 16
    check_against_oracle(x_host, group, x_dev=x_dev, label="16B-aligned")


# ---------------------------------------------------------------- beyond 32-bit indices -----

@pytest.mark.parametrize("group", [16, 256])
def test_more_than_2_pow_32_elements(group):
    """bf16 [65537, 65536]: 2^32 + 65536 elements (8.6 GB), so element and byte offsets pass
    2^32 and 2^33.  Every value lies in [-1, 1) except one planted 1024 in the last row: any
    other rotation group has |y| < 16 (at most G values under 1, times 1/sqrt(G)), while the
    planted group has max |y| >= 64 (the rotation is orthonormal), so the tensor's amax is the
    last row's, which the oracle computes.  Rows on both sides of element 2^32 and a few others
    are then compared with the oracle byte for byte (codes, scales, and the scales of the
    swizzled pass at their tile positions), with that amax; so are MXFP4's codes and scales
    (no global scale)."""
    M, K = 65537, 65536
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev)
    gen.manual_seed(2024 + group)
    x = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    for r0 in range(0, M, 4096):
        r1 = min(M, r0 + 4096)
        x[r0:r1] = (torch.rand((r1 - r0, K), generator=gen, device=dev) * 2 - 1).to(torch.bfloat16)
    x[M - 1, K - 200] = 1024.0
    amax = hq.hq_rot_amax(x, group)
    q, s, sg = hq.hq_rotate_quant_nvfp4(x, group, amax)
    torch.cuda.synchronize()
    rows = [0, 1, 12345, 32768, 65534, 65535, 65536]   # row 65536 starts at element 2^32
    xs = synth.as_oracle_array(x[rows].cpu())
    _, _, last_amax, _ = oracle.quantize(xs[-1:], group)
    assert f32_bits(amax.cpu().numpy())[0] == f32_bits([last_amax])[0]
    oq, os_, _, osg = oracle.quantize(xs, group, amax=float(last_amax))
    assert f32_bits(sg.cpu().numpy())[0] == f32_bits([osg])[0]
    assert_bytes_equal("scales", s[rows].cpu().numpy(), os_)
    assert_bytes_equal("codes", q[rows].cpu().numpy(), oq)
    # swizzled scales: row r, column c at 512 (r / 128 * col_tiles + c / 4) + (r % 32) 16 +
    # (r / 32 % 4) 4 + c % 4 of the padded buffer
    del s
    s_sw = torch.empty(hq.hq_swizzled_scales_bytes(M, K), dtype=torch.uint8, device=dev)
    q.fill_(0)
    hq.hq_rotate_quant_nvfp4_swizzled(x, group, amax, q=q, scales=s_sw)
    torch.cuda.synchronize()
    col_tiles = (K // 16 + 3) // 4
    c = np.arange(K // 16)
    offs = np.stack([512 * ((r // 128) * col_tiles + c // 4) + (r % 32) * 16 + (r // 32 % 4) * 4 + c % 4
                     for r in rows])
    got = s_sw.cpu().numpy()[offs]
    assert_bytes_equal("swizzled scales", got, os_)
    assert_bytes_equal("swizzled-pass codes", q[rows].cpu().numpy(), oq)
    del s_sw
    smx = torch.empty((M, K // 32), dtype=torch.uint8, device=dev)
    hq.hq_rotate_quant_mxfp4(x, group, q=q, scales=smx)
    torch.cuda.synchronize()
    mq, ms = oracle.quantize_mxfp4(xs, group)
    assert_bytes_equal("mxfp4 scales", smx[rows].cpu().numpy(), ms)
    assert_bytes_equal("mxfp4 codes", q[rows].cpu().numpy(), mq)
