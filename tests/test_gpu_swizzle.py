"""Swizzled block scales (hq_rotate_quant_nvfp4_swizzled, _ws) against the oracle, and as the input of
cuBLASLt's NVFP4 GEMM.

"A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §6 "From interpreter to hardware"
(Layout): GEMM consumers read the block scales in a swizzled tiled layout, which a production
kernel writes directly.  The codes and s_global equal pass 2's; the scales equal the oracle's
row-major scales moved by oracle.swizzle_scales, padding written as zeros.  The consumer test feeds
codes and swizzled scales of two tensors to torch._scaled_mm (cuBLASLt, NVFP4 with E4M3 block
scales) and compares the product with the oracle's dequantized tensors multiplied in float64:
a misplaced scale would scale a 16-element slice of a dot product by a wrong power.
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


def varied(M, K, seed, dtype=torch.bfloat16):
    """Rows and 16-blocks at different magnitudes, so that block scales differ widely."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2((np.arange(M) % 7) - 3.0).astype(np.float32)[:, None]
    x *= np.exp2(((np.arange(K) // 16) % 5) - 2.0).astype(np.float32)[None, :]
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def run_swizzled(x_host, group, x_dev=None):
    x = x_dev if x_dev is not None else x_host.cuda()
    amax = hq.hq_rot_amax(x, group)
    q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled(x, group, amax)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), sg.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 16), (3, 48), (128, 64), (129, 80), (200, 96), (300, 1040),
                                 (1024, 4096)])
@pytest.mark.parametrize("group", [0, 16, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_swizzled_parity(M, K, group, dtype):
    if group == 256 and K % 256:
        pytest.skip("K not a multiple of 256")
    x = varied(M, K, seed=M + K + group, dtype=dtype)
    q, s, sg = run_swizzled(x, group)
    oq, os_, _, osg = oracle.quantize(synth.as_oracle_array(x), group)
    assert np.array_equal(q, oq)
    assert np.array_equal(sg.view(np.uint32), np.array([osg], np.float32).view(np.uint32))
    assert np.array_equal(s, oracle.swizzle_scales(os_))   # padding stays zero too


@pytest.mark.parametrize("group", [0, 16, 256])
def test_every_byte_of_the_swizzled_buffer_is_written(group):
    M, K = 131, 512 + 48 * (group != 256)
    x = varied(M, K, seed=5)
    xd = x.cuda()
    amax = hq.hq_rot_amax(xd, group)
    s = torch.full((hq.hq_swizzled_scales_bytes(M, K),), 0xFF, dtype=torch.uint8, device="cuda")
    q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled(xd, group, amax, scales=s)
    _, os_, _, _ = oracle.quantize(synth.as_oracle_array(x), group)
    assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


@pytest.mark.parametrize("group", [16, 256])
def test_swizzled_strided_rows(group):
    big = varied(160, 512 + 64, seed=3)
    x = big[:, :512].contiguous()
    q, s, sg = run_swizzled(x, group, x_dev=big.cuda()[:, :512])
    oq, os_, _, _ = oracle.quantize(synth.as_oracle_array(x), group)
    assert np.array_equal(q, oq) and np.array_equal(s, oracle.swizzle_scales(os_))


# hq_rotate_quant_nvfp4_swizzled_ws: the units (8 rows x 128 blocks) are handed out at run time
# from 16384 tiles (2048 units) on; below that it is the fixed split.  Twice on one workspace.
@pytest.mark.parametrize("M,K,group,dtype", [(129, 80, 16, torch.bfloat16), (4099, 8192, 16, torch.bfloat16),
                                             (2053, 17408, 16, torch.bfloat16), (4099, 8192, 256, torch.bfloat16),
                                             (2053, 17408, 0, torch.bfloat16), (4099, 8192, 16, torch.float32),
                                             (2053, 17408, 256, torch.float32)])
def test_swizzled_with_a_workspace(M, K, group, dtype):
    if K % max(group, 16):
        pytest.skip("K not a multiple of the group")
    x = varied(M, K, seed=M + K + group, dtype=dtype)
    xd = x.cuda()
    oq, os_, _, osg = oracle.quantize(synth.as_oracle_array(x), group)
    amax = hq.hq_rot_amax(xd, group)
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    for _ in range(2):
        s = torch.full((hq.hq_swizzled_scales_bytes(M, K),), 0xFF, dtype=torch.uint8, device="cuda")
        q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled_ws(xd, group, amax, scales=s, workspace=ws)
        torch.cuda.synchronize()
        assert not ws.any().item(), "the workspace is not back to 0"
        assert np.array_equal(q.cpu().numpy(), oq)
        assert np.array_equal(sg.cpu().numpy().view(np.uint32), np.array([osg], np.float32).view(np.uint32))
        assert np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


def test_swizzled_with_a_workspace_strided_rows():
    big = varied(4099, 8192 + 64, seed=4)
    x = big[:, :8192].contiguous()
    xd = big.cuda()[:, :8192]
    oq, os_, _, _ = oracle.quantize(synth.as_oracle_array(x), 16)
    amax = hq.hq_rot_amax(xd, 16)
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled_ws(xd, 16, amax, workspace=ws)
    torch.cuda.synchronize()
    assert not ws.any().item()
    assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), oracle.swizzle_scales(os_))


def _nvfp4_gemm(qa, sa, qb, sb):
    """cuBLASLt NVFP4 GEMM through torch: A [M, K] (codes [M, K/2]) times B^T (B [N, K])."""
    a = qa.view(torch.float4_e2m1fn_x2)
    b = qb.view(torch.float4_e2m1fn_x2).t()
    sa8 = sa.view(torch.float8_e4m3fn)
    sb8 = sb.view(torch.float8_e4m3fn)
    errors = []
    for out in (torch.float32, torch.bfloat16):
        try:
            return torch._scaled_mm(a, b, sa8, sb8, out_dtype=out).float(), out
        except (RuntimeError, NotImplementedError, TypeError) as e:
            if "Invalid blockwise scaling" in str(e):
                raise
            errors.append(f"{out}: {str(e).splitlines()[0][:160]}")
    pytest.skip("NVFP4 GEMM not available in this torch / cuBLASLt: " + " | ".join(errors))


@pytest.mark.parametrize("M,N,K", [(200, 144, 96), (256, 128, 1024), (384, 256, 2048)])
def test_cublaslt_nvfp4_gemm_reads_the_swizzled_scales(M, N, K):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no float4_e2m1fn_x2")
    xa = varied(M, K, seed=11 + K)
    xb = varied(N, K, seed=12 + K)
    res = {}
    for name, x in (("a", xa), ("b", xb)):
        xd = x.cuda()
        amax = hq.hq_rot_amax(xd, 16)
        q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled(xd, 16, amax)
        res[name] = (q, s, float(sg.item()))
    got, out_dtype = _nvfp4_gemm(res["a"][0], res["a"][1], res["b"][0], res["b"][1])
    got = got.cpu().double().numpy() * res["a"][2] * res["b"][2]
    # reference: the oracle's dequantized tensors (same codes and scales), multiplied in float64
    da = oracle.dequant(res["a"][0].cpu().numpy(), oracle.unswizzle_scales(res["a"][1].cpu().numpy(), M, K // 16),
                        res["a"][2], 16, False).astype(np.float64)
    db = oracle.dequant(res["b"][0].cpu().numpy(), oracle.unswizzle_scales(res["b"][1].cpu().numpy(), N, K // 16),
                        res["b"][2], 16, False).astype(np.float64)
    ref = da @ db.T
    mag = np.abs(da) @ np.abs(db).T
    # fp32 accumulation of up to 2048 products: far below 2^-12 of sum |a b|; one misplaced
    # 16-block scale moves a result by about 2^-7 of it or more (K <= 2048, scales 2x apart)
    rel = 2.0 ** -12 if out_dtype == torch.float32 else 2.0 ** -7
    assert np.all(np.abs(got - ref) <= rel * mag + 1e-30), np.max(np.abs(got - ref) / (mag + 1e-30))
