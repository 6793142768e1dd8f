"""MXFP4 (hq_rotate_quant_mxfp4, hq_rotate_quant_mxfp4_ws / hq_dequant_mxfp4) against the oracle,
bit-exact.

"A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §1 (MXFP4: 32-element blocks, E8M0
power-of-two scales) and "Try this" (the error study with MXFP4 semantics); scale rule as the
oracle documents.
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
    x[:, rng.choice(K, max(1, K // 64), replace=False)] *= 30.0
    if M > 3:
        x[2] = 0.0
        x[3, : K // 2] *= np.float32(1e-36)
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def check(x_host, group, x_dev=None, roundtrip=False, ws=None):
    x = x_dev if x_dev is not None else x_host.cuda()
    if ws is None:
        q, s = hq.hq_rotate_quant_mxfp4(x, group)
    else:
        q, s = hq.hq_rotate_quant_mxfp4_ws(x, group, workspace=ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert not ws.any().item(), "the workspace is not back to 0"
    xo = synth.as_oracle_array(x_host)
    oq, os_ = oracle.quantize_mxfp4(xo, group)
    assert np.array_equal(s.cpu().numpy(), os_), "scales differ"
    gq = q.cpu().numpy()
    if not np.array_equal(gq, oq):
        bad = np.argwhere(gq != oq)
        raise AssertionError(f"{len(bad)} code bytes differ, first {bad[:5].tolist()}")
    if roundtrip:
        for un in ([False, True] if group else [False]):
            back = hq.hq_dequant_mxfp4(q, s, group if group else 16, un)
            torch.cuda.synchronize()
            ref = oracle.dequant_mxfp4(oq, os_, group, un)
            assert np.array_equal(back.cpu().numpy().view(np.uint32), ref.view(np.uint32))


SHAPES = [(1, 32, 0), (1, 32, 16), (2, 256, 256), (17, 96, 16), (129, 256, 256), (1000, 288, 0),
          (257, 1024, 16), (31, 4096, 256), (4099, 64, 16)]


@pytest.mark.parametrize("M,K,group", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mxfp4_parity(M, K, group, dtype):
    check(rand_input(M, K, dtype, seed=M + K + group), group, roundtrip=True)


@pytest.mark.parametrize("group", [0, 16, 256])
def test_mxfp4_strided(group):
    big = rand_input(300, 1280, torch.bfloat16, seed=6)
    check(big[:, :1024].contiguous(), group, x_dev=big.cuda()[:, :1024])


@pytest.mark.parametrize("scale_exp", [-140, -126, -110, 60, 110])
@pytest.mark.parametrize("group", [0, 16, 256])
def test_mxfp4_extreme_magnitudes(scale_exp, group):
    x = (rand_input(40, 512, torch.float32, seed=abs(scale_exp)).double() * 2.0 ** scale_exp).float()
    check(x, group, roundtrip=True)


@pytest.mark.parametrize("name", ["bf16_16384x8192_t3", "bf16_8192x16384_g256"])
def test_mxfp4_on_named_workloads(name):
    w = synth.WORKLOADS[name]
    x = synth.generate(w)
    check(x, w.groups[0])


def new_workspace():
    return torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")


# hq_rotate_quant_mxfp4_ws: the tiles are handed out at run time from 16384 warp tiles on
# (2^21 16-blocks); below that, and for strided rows, it is the fixed split.
@pytest.mark.parametrize("M,K,group", [(1, 32, 16), (999, 4352, 16), (4099, 8192, 16), (16385, 2048, 256),
                                       (2053, 17408, 0), (4099, 8192, 256)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mxfp4_with_a_workspace(M, K, group, dtype):
    x = rand_input(M, K, dtype, seed=M + 3 * K + group)
    ws = new_workspace()
    for _ in range(2):  # twice on one workspace: the first call leaves it ready for the next
        check(x, group, ws=ws)


def test_mxfp4_with_a_workspace_strided():
    big = rand_input(300, 1280, torch.bfloat16, seed=9)
    check(big[:, :1024].contiguous(), 16, x_dev=big.cuda()[:, :1024], ws=new_workspace())


def test_mxfp4_with_a_workspace_on_the_named_workload():
    w = synth.WORKLOADS["bf16_16384x8192_t3"]
    check(synth.generate(w), 16, ws=new_workspace())
