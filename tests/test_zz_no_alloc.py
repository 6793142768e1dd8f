"""The allocation-free entry point, hq_quantize_nvfp4_host_noalloc.

It serves callers that cannot allocate device memory: for example a plug-in inside a host
program that owns the device memory pool, or a serving loop whose memory footprint is fixed
at start-up.  Instead of a workspace, it stages the tensor in a fixed array inside the library.
These tests call it through the C ABI on two calls in a row, with different tensors, rotation
groups and sizes, so that a second call cannot lean on what the first left in the shared array.
Each result must equal, byte for byte, what the existing entry points (hq_rot_amax and
hq_rotate_quant_nvfp4 on device buffers) produce for the same input, and what the CPU oracle
computes from the definition.  A tensor larger than the array must be refused before anything
runs.

This file is collected last on purpose; it needs no state from the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import hadamard_rotation_gb300 as hq
import oracle
from hadamard_rotation_gb300 import synth

pytestmark = pytest.mark.gpu

HQ_OK = 0
HQ_ERR_TOO_LARGE = 7
NOALLOC_BYTES = 32 * 1024 * 1024  # HQ_NOALLOC_SCRATCH_BYTES in include/hq.h


@pytest.fixture(scope="module")
def lib():
    from hadamard_rotation_gb300 import build

    build.build()
    oracle.build()
    lib = hq.load()
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.hq_quantize_nvfp4_host_noalloc.argtypes = [p, i32, i64, i64, i32, p, p, p, p]
    lib.hq_quantize_nvfp4_host_noalloc.restype = i32
    return lib


def host_input(M, K, dtype, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x[:, rng.choice(K, K // 64, replace=False)] *= 40.0
    x[3] = 0.0
    t = torch.from_numpy(x)
    return (t if dtype == torch.float32 else t.to(dtype)).pin_memory()


def noalloc(lib, x_host, group):
    M, K = x_host.shape
    q = torch.empty((M, K // 2), dtype=torch.uint8, pin_memory=True)
    s = torch.empty((M, K // 16), dtype=torch.uint8, pin_memory=True)
    sg = torch.empty(1, dtype=torch.float32, pin_memory=True)
    dt = 1 if x_host.dtype == torch.bfloat16 else 0
    stream = torch.cuda.current_stream()
    rc = lib.hq_quantize_nvfp4_host_noalloc(
        ctypes.c_void_p(x_host.data_ptr()), dt, M, K, group, ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(sg.data_ptr()),
        ctypes.c_void_p(stream.cuda_stream))
    assert rc == HQ_OK, lib.hq_status_string(rc)
    stream.synchronize()
    return q.numpy().copy(), s.numpy().copy(), sg.numpy().copy()


def existing(x_host, group):
    x = x_host.cuda()
    amax = hq.hq_rot_amax(x, group)
    q, s, sg = hq.hq_rotate_quant_nvfp4(x, group, amax)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy(), sg.cpu().numpy()


def test_noalloc_matches_existing_entry_points_on_two_calls_in_a_row(lib):
    cases = [(2048, 4096, torch.bfloat16, 16, 1),   # about 8.4 M elements
             (300, 1024, torch.float32, 256, 2)]     # smaller, other dtype and group
    for M, K, dtype, group, seed in cases:
        x_host = host_input(M, K, dtype, seed)
        got = noalloc(lib, x_host, group)
        ref = existing(x_host, group)
        oq, os_, _, osg = oracle.quantize(synth.as_oracle_array(x_host), group)
        defined = (oq, os_, np.array([osg], np.float32))
        for name, g, r, o in zip(("codes", "scales", "s_global"), got, ref, defined):
            assert np.array_equal(g.view(np.uint8), r.view(np.uint8)), (name, M, K, group)
            assert np.array_equal(g.view(np.uint8), o.view(np.uint8)), (name, M, K, group, "oracle")


def test_noalloc_refuses_a_tensor_larger_than_its_scratch(lib):
    M, K = 4096, 4096  # 16.8 M bf16 elements: needs about 43 MB of the 32 MiB array
    x = torch.empty(1, dtype=torch.bfloat16, pin_memory=True)
    out = torch.empty(1, dtype=torch.uint8, pin_memory=True)
    rc = lib.hq_quantize_nvfp4_host_noalloc(
        ctypes.c_void_p(x.data_ptr()), 1, M, K, 16, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(out.data_ptr()), None)
    assert rc == HQ_ERR_TOO_LARGE
    assert b"TOO_LARGE" in lib.hq_status_string(rc)
