"""Single-pass, delayed-amax mode (hq_rotate_quant_nvfp4_delayed, _ws) against the oracle.

"A Fused Hadamard + NVFP4 Quantization Kernel in Triton", §2: production stacks may reuse an amax
from a previous step so that the per-block work is a single pass.  The oracle side is the same
definition with the given amax (oracle.quantize(..., amax=prev)) plus the tensor's own amax
(oracle.rot_amax).  Everything must be bit-exact.
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


def bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


def rand_input(M, K, dtype, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, rng.choice(K, max(1, K // 64), replace=False)] *= 30.0
    x[1] = 0.0
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def check(x_host, group, prev, x_dev=None, ws=None):
    x = x_dev if x_dev is not None else x_host.cuda()
    a_prev = torch.tensor([prev], dtype=torch.float32, device=x.device)
    if ws is None:
        q, s, sg, a_next = hq.hq_rotate_quant_nvfp4_delayed(x, group, a_prev)
    else:
        a_next = torch.full((1,), 7.0, dtype=torch.float32, device=x.device)  # overwritten
        q, s, sg, a_next = hq.hq_rotate_quant_nvfp4_delayed_ws(x, group, a_prev, amax_next=a_next,
                                                               workspace=ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert not ws.any().item(), "the workspace is not back to 0"
    xo = synth.as_oracle_array(x_host)
    oq, os_, _, osg = oracle.quantize(xo, group, amax=float(np.float32(prev)))
    oamax, _ = oracle.rot_amax(xo, group)
    assert bits(a_next.cpu().numpy())[0] == bits([oamax])[0]
    assert bits(sg.cpu().numpy())[0] == bits([osg])[0]
    assert np.array_equal(s.cpu().numpy(), os_)
    assert np.array_equal(q.cpu().numpy(), oq)
    return oamax


@pytest.mark.parametrize("group", [0, 16, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_delayed_equals_definition_with_the_given_amax(group, dtype):
    x = rand_input(333, 1024, dtype, seed=group + 7)
    true_amax = check(x, group, 1.0)
    # exact amax: the two-pass result; stale (smaller) amax: saturating scales; larger amax
    for prev in (true_amax, true_amax * 0.3, true_amax * 0.9999, true_amax * 4.0, 1e-30, 1e30, 0.0):
        check(x, group, prev)


def test_delayed_with_exact_amax_equals_two_pass_on_a_workload():
    w = synth.WORKLOADS["bf16_16384x8192_t3"]
    x_host = synth.generate(w)
    x = x_host.cuda()
    amax = hq.hq_rot_amax(x, 16)
    q2, s2, sg2 = hq.hq_rotate_quant_nvfp4(x, 16, amax)
    q1, s1, sg1, a_next = hq.hq_rotate_quant_nvfp4_delayed(x, 16, amax)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(s1, s2) and torch.equal(sg1, sg2)
    assert torch.equal(a_next, amax)
    check(x_host, 16, float(amax.item()) * 0.5, x_dev=x)


def test_delayed_strided_rows():
    big = rand_input(200, 1280, torch.bfloat16, seed=3)
    x_dev = big.cuda()[:, :1024]
    check(big[:, :1024].contiguous(), 256, 5.0, x_dev=x_dev)


def test_delayed_steps_chain():
    """Step t quantizes with the amax reduced in step t-1, on a sequence of tensors."""
    prev = torch.zeros(1, dtype=torch.float32, device="cuda")
    for t in range(4):
        x_host = rand_input(128, 512, torch.bfloat16, seed=40 + t) * (1.0 + t)
        x = x_host.cuda()
        expect_prev = float(prev.item())
        q, s, sg, nxt = hq.hq_rotate_quant_nvfp4_delayed(x, 16, prev)
        torch.cuda.synchronize()
        oq, os_, _, _ = oracle.quantize(synth.as_oracle_array(x_host), 16, amax=expect_prev)
        assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), os_)
        prev = nxt.clone()


def test_delayed_surfaces_nonfinite_in_next_amax():
    x = torch.ones(64, 512, device="cuda")
    a = torch.ones(1, device="cuda")
    x[3, 3] = float("inf")
    for g in (0, 16, 256):
        assert torch.isinf(hq.hq_rotate_quant_nvfp4_delayed(x, g, a)[3]).item()
    x[9, 100] = float("nan")
    for g in (0, 16, 256):
        assert torch.isnan(hq.hq_rotate_quant_nvfp4_delayed(x, g, a)[3]).item()


def test_delayed_rejects_aliased_amax():
    x = torch.ones(4, 32, device="cuda")
    a = torch.ones(1, device="cuda")
    with pytest.raises(hq.HQError):
        hq.hq_rotate_quant_nvfp4_delayed(x, 16, a, amax_next=a)


# hq_rotate_quant_nvfp4_delayed_ws: the next amax reduced in the workspace (no memset), the tiles
# handed out at run time from 16384 tiles on; twice on one workspace.
@pytest.mark.parametrize("M,K,group", [(333, 1024, 16), (4099, 8192, 16), (16385, 2048, 256), (2053, 17408, 0)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_delayed_with_a_workspace(M, K, group, dtype):
    x = rand_input(M, K, dtype, seed=M + K + group)
    xd = x.cuda()
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    true_amax = check(x, group, 1.0, x_dev=xd, ws=ws)
    check(x, group, true_amax, x_dev=xd, ws=ws)
    check(x, group, true_amax * 0.3, x_dev=xd, ws=ws)


def test_delayed_with_a_workspace_strided_rows():
    big = rand_input(4099, 8192 + 64, torch.bfloat16, seed=5)
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    check(big[:, :8192].contiguous(), 16, 2.5, x_dev=big.cuda()[:, :8192], ws=ws)
