"""The paths bench.py times, checked against the oracle on the bench tensor itself (bf16
[32768, 28672], the 1.88 GB LLM MLP-up-sized workload) in the launch configuration the bench
uses:

  - the metric's step verbatim: hq_quantize_nvfp4 with a workspace, which on this tensor is the
    streaming pass 1 reducing into the workspace (its last CTA writes amax) and pass 2, both
    launched as programmatic dependents; twice in a row on one workspace;
  - delayed-amax single pass with the true amax: codes and scales equal pass 2's, the amax it
    reduces equals the tensor's;
  - pass 2 with swizzled scales: codes in full; the scales of sampled 128-row tiles (first,
    middle, last) equal the oracle's row-major scales of those rows, re-indexed;
  - MXFP4, group 16: codes and E8M0 scales in full;
  - INT8 per token, group 256 (14 warp tiles per row here): codes and row scales in full.
"""
import numpy as np
import pytest
import torch

import hadamard_rotation_gb300 as hq
import oracle
from hadamard_rotation_gb300 import synth

pytestmark = pytest.mark.gpu

NAME = "bf16_32768x28672"


@pytest.fixture(scope="module")
def bench_tensor():
    from hadamard_rotation_gb300 import build

    build.build()
    oracle.build()
    hq.load()
    x_host = synth.generate(synth.WORKLOADS[NAME])
    return x_host, x_host.cuda(), synth.as_oracle_array(x_host)


@pytest.fixture(scope="module")
def nvfp4_reference(bench_tensor):
    _, _, xo = bench_tensor
    return oracle.quantize(xo, 16)


# A finished call leaves every workspace word 0 (the next call relies on it).
def settled(ws) -> bool:
    return not ws.any().item()


def f32_bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def test_bench_step_twice_on_one_workspace(bench_tensor, nvfp4_reference):
    _, x, _ = bench_tensor
    oq, os_, oamax, osg = nvfp4_reference
    M, K = x.shape
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    amax = torch.empty(1, dtype=torch.float32, device="cuda")
    q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    s = torch.empty((M, K // 16), dtype=torch.uint8, device="cuda")
    sg = torch.empty(1, dtype=torch.float32, device="cuda")
    for call in range(2):
        q.fill_(0xEE)
        s.fill_(0xEE)
        hq.hq_quantize_nvfp4(x, 16, amax=amax, q=q, scales=s, s_global=sg, workspace=ws)
        torch.cuda.synchronize()
        assert f32_bits(amax.cpu().numpy())[0] == f32_bits([oamax])[0], call
        assert f32_bits(sg.cpu().numpy())[0] == f32_bits([osg])[0], call
        assert np.array_equal(s.cpu().numpy(), os_), call
        assert np.array_equal(q.cpu().numpy(), oq), call
        assert settled(ws), call         # the workspace is ready for the next call
    assert hq.hq_read_fault() == 0


def test_delayed_single_pass(bench_tensor, nvfp4_reference):
    _, x, _ = bench_tensor
    oq, os_, oamax, osg = nvfp4_reference
    amax = torch.tensor([oamax], dtype=torch.float32, device="cuda")
    q, s, sg, amax_next = hq.hq_rotate_quant_nvfp4_delayed(x, 16, amax)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), os_)
    assert f32_bits(sg.cpu().numpy())[0] == f32_bits([osg])[0]
    assert f32_bits(amax_next.cpu().numpy())[0] == f32_bits([oamax])[0]


def test_swizzled_scales(bench_tensor, nvfp4_reference):
    _, x, _ = bench_tensor
    oq, os_, _, _ = nvfp4_reference
    amax = hq.hq_rot_amax(x, 16)
    q, s, sg = hq.hq_rotate_quant_nvfp4_swizzled(x, 16, amax)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), oq)
    buf = s.cpu().numpy()
    M, C0 = os_.shape
    tile_row_bytes = 128 * (-(-C0 // 4) * 4)       # one 128-row tile of the swizzled layout
    for t in (0, (M // 128) // 2, M // 128 - 1):
        got = buf[t * tile_row_bytes:(t + 1) * tile_row_bytes]
        assert np.array_equal(got, oracle.swizzle_scales(os_[128 * t:128 * (t + 1)])), t


def test_mxfp4(bench_tensor):
    _, x, xo = bench_tensor
    q, s = hq.hq_rotate_quant_mxfp4(x, 16)
    torch.cuda.synchronize()
    oq, os_ = oracle.quantize_mxfp4(xo, 16)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy(), os_)


def test_int8_per_token_group_256(bench_tensor):
    _, x, xo = bench_tensor
    q, sc = hq.hq_rotate_quant_int8(x, 256)
    torch.cuda.synchronize()
    oq, osc = oracle.rotate_quant_int8(xo, 256)
    assert np.array_equal(f32_bits(sc.cpu().numpy()), f32_bits(osc))
    gq = q.cpu().numpy()
    if not np.array_equal(gq, oq):
        bad = np.argwhere(gq != oq)
        raise AssertionError(f"{len(bad)} int8 codes differ, first {bad[:5].tolist()}")
