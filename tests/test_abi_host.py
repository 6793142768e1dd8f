"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports every
function include/hq.h declares, and rejects bad arguments synchronously, before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hq.h")

FAKE = 0x10000  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    from hadamard_rotation_gb300 import build
    import hadamard_rotation_gb300 as hq

    build.build()
    return hq.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("hq_rot_amax", "hq_rotate_quant_nvfp4", "hq_dequant_nvfp4"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "hq.h"\nint main(void){ return (int)HQ_OK + (int)HQ_BF16; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c",
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_a_c_program_links_and_calls_the_library(tmp_path, lib):
    """The boundary from C itself: a C99 program built with gcc against include/hq.h and
    linked to libhq.so calls entry points whose arguments fail validation (no GPU needed)
    and reads the status strings."""
    src = tmp_path / "caller.c"
    src.write_text(r"""
#include <stdio.h>
#include "hq.h"
int main(void) {
  float amax;
  unsigned char q[64], s[16];
  unsigned int ws[HQ_QUANTIZE_WORKSPACE_WORDS];
  hq_status a = hq_rot_amax(NULL, HQ_BF16, 4, 64, 64, 16, &amax, NULL, NULL);
  hq_status b = hq_rotate_quant_nvfp4((const void*)q, HQ_BF16, 4, 64, 64, 32, &amax, q, s, NULL, NULL);
  hq_status c = hq_quantize_nvfp4((const void*)q, HQ_BF16, 4, 24, 24, 16, &amax, q, s, NULL, ws, NULL);
  hq_status d = hq_rotate_quant_mxfp4_ws((const void*)q, HQ_BF16, 4, 48, 48, 16, q, s, ws, NULL);
  hq_status e = hq_rotate_quant_nvfp4_ws((const void*)q, HQ_BF16, 0, 64, 64, 16, &amax, q, s, NULL, ws, NULL);
  printf("%d %d %d %d %d %d\n", (int)a, (int)b, (int)c, (int)d, (int)e, hq_version());
  printf("%s\n", hq_status_string(a));
  return 0;
}
""")
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib._name)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), str(src),
                    "-L", libdir, "-lhq", "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    assert out[0].split() == ["1", "5", "2", "2", "0", "100"]   # NULL x, group 32, K % 16, K % 32, M = 0
    assert out[1].startswith("HQ_ERR_NULL")


def test_version_and_status_strings(lib):
    assert lib.hq_version() >= 100
    for code in range(9):
        assert lib.hq_status_string(code).decode().startswith("HQ_")
    assert b"unknown" in lib.hq_status_string(99)
    assert lib.hq_last_cuda_error() == 0


P = ctypes.c_void_p


def rq(lib, x=FAKE, dt=1, M=4, K=32, ldx=32, G=16, amax=FAKE, q=FAKE, s=FAKE, sg=None):
    return lib.hq_rotate_quant_nvfp4(P(x) if x else None, dt, M, K, ldx, G, P(amax) if amax else None,
                                     P(q) if q else None, P(s) if s else None,
                                     P(sg) if sg else None, None)


def ra(lib, x=FAKE, dt=1, M=4, K=32, ldx=32, G=16, amax=FAKE, y=None):
    return lib.hq_rot_amax(P(x) if x else None, dt, M, K, ldx, G, P(amax) if amax else None,
                           P(y) if y else None, None)


def dq(lib, q=FAKE, s=FAKE, sg=FAKE, M=4, K=32, G=16, un=1, out=FAKE):
    return lib.hq_dequant_nvfp4(P(q) if q else None, P(s) if s else None, P(sg) if sg else None,
                                M, K, G, un, P(out) if out else None, None)


def test_null_pointers(lib):
    assert rq(lib, x=0) == 1 and rq(lib, amax=0) == 1 and rq(lib, q=0) == 1 and rq(lib, s=0) == 1
    assert ra(lib, x=0) == 1 and ra(lib, amax=0) == 1
    assert dq(lib, q=0) == 1 and dq(lib, s=0) == 1 and dq(lib, sg=0) == 1 and dq(lib, out=0) == 1


def test_bad_shapes(lib):
    assert rq(lib, K=24, ldx=24) == 2            # K not a multiple of 16
    assert rq(lib, K=272, ldx=272, G=256) == 2   # K not a multiple of 256
    assert rq(lib, M=-1) == 2
    assert rq(lib, K=-16) == 2
    assert rq(lib, ldx=16) == 2                  # ldx < K
    assert rq(lib, M=2 ** 62, K=64, ldx=64) == 2  # M*K overflows
    big = 2 ** 36                                 # 2^32 blocks in one row: beyond the kernels
    assert rq(lib, M=1, K=big, ldx=big) == 2 and ra(lib, M=1, K=big, ldx=big) == 2
    assert lib.hq_rotate_quant_mxfp4(P(FAKE), 1, 1, big, big, 16, P(FAKE), P(FAKE), None) == 2
    assert lib.hq_quantize_nvfp4(P(FAKE), 1, 1, big, big, 16, P(FAKE), P(FAKE), P(FAKE), None,
                                 P(FAKE + 256), None) == 2
    if not torch.cuda.is_available():             # one block less passes the shape checks
        assert ra(lib, M=1, K=big - 16, ldx=big - 16) == 6
    assert ra(lib, K=48, ldx=48, G=256) == 2
    assert dq(lib, K=24) == 2
    assert dq(lib, K=272, G=256) == 2
    assert dq(lib, M=-3) == 2


def test_bad_group_and_dtype(lib):
    for G in (1, 8, 32, 64, 128, 512, -16):
        assert rq(lib, G=G) == 5 and ra(lib, G=G) == 5
    assert dq(lib, G=0, un=1) == 5
    assert dq(lib, G=32, un=0) == 5
    assert rq(lib, dt=2) == 4 and ra(lib, dt=-1) == 4


def test_alignment(lib):
    assert rq(lib, x=FAKE + 2) == 3
    assert rq(lib, dt=1, ldx=36) == 3            # 72 B row stride: not a multiple of 16
    assert rq(lib, dt=0, ldx=34) == 3            # 136 B row stride
    assert rq(lib, q=FAKE + 8) == 3
    assert rq(lib, s=FAKE + 2) == 3
    assert rq(lib, amax=FAKE + 2) == 3
    assert rq(lib, sg=FAKE + 1) == 3
    assert ra(lib, y=FAKE + 4) == 3
    assert dq(lib, out=FAKE + 8) == 3
    assert dq(lib, q=FAKE + 4) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a CUDA device")
def test_valid_arguments_without_a_device_report_cuda_error(lib):
    # Arguments pass validation, so the call reaches the CUDA runtime, which has no device.
    assert ra(lib) == 6
    assert lib.hq_last_cuda_error() != 0


def test_empty_quantize_is_a_noop(lib):
    # M == 0: valid, nothing to enqueue (no CUDA call is made for pass 2 or dequant).
    assert rq(lib, M=0) == 0
    assert dq(lib, M=0) == 0


def test_binding_rejects_host_tensors():
    import hadamard_rotation_gb300 as hq

    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        hq.hq_rot_amax(x, 16)
    with pytest.raises(ValueError, match="CUDA"):
        hq.hq_rotate_quant_nvfp4(x, 16, torch.zeros(1))


def test_binding_refuses_a_stream_of_another_device():
    # The library launches on the current device; the binding makes the tensors' device
    # current and must not hand it a stream that belongs to another device.
    from hadamard_rotation_gb300 import api

    class FakeStream:
        device = torch.device("cuda", 1)
        cuda_stream = 0

    with pytest.raises(ValueError, match="stream is on cuda:1"):
        api._stream_handle(FakeStream(), torch.device("cuda", 0))
    assert api._stream_handle(FakeStream(), torch.device("cuda", 1)).value is None  # handle 0


def test_read_fault_rejects_null(lib):
    assert lib.hq_read_fault(None, 0) == 1


def test_host_pipeline_argument_checks(lib):
    PP = ctypes.POINTER(ctypes.c_void_p)
    out = ctypes.c_void_p(1234)
    ref = ctypes.byref(out)
    assert lib.hq_host_pipeline_workspace_bytes(0, 32, 1) == 0
    assert lib.hq_host_pipeline_workspace_bytes(4, 24, 1) == 0
    assert lib.hq_host_pipeline_workspace_bytes(4, 32, 7) == 0
    assert lib.hq_host_pipeline_workspace_bytes(2 ** 40, 2 ** 22, 0) == 0   # bytes would wrap
    assert lib.hq_host_pipeline_workspace_bytes(1, 2 ** 36, 1) == 0        # row too long
    assert lib.hq_host_pipeline_create(1, 2 ** 36, 1, 16, P(FAKE), 2 ** 40, ref) == 2
    need = lib.hq_host_pipeline_workspace_bytes(4, 32, 1)
    assert need > 2 * (4 * 32 * 2)
    assert lib.hq_host_pipeline_create(4, 32, 1, 16, None, need, ref) == 1
    assert out.value is None or out.value == 1234 or out.value == 0
    assert lib.hq_host_pipeline_create(4, 32, 1, 16, P(FAKE), need, None) == 1
    assert lib.hq_host_pipeline_create(4, 32, 5, 16, P(FAKE), need, ref) == 4
    assert lib.hq_host_pipeline_create(4, 32, 1, 8, P(FAKE), need, ref) == 5
    assert lib.hq_host_pipeline_create(4, 48, 1, 256, P(FAKE), need, ref) == 2
    assert lib.hq_host_pipeline_create(4, 32, 1, 16, P(FAKE + 16), need, ref) == 3
    assert lib.hq_host_pipeline_create(4, 32, 1, 16, P(FAKE), need - 1, ref) == 2
    assert lib.hq_host_pipeline_submit(None, P(FAKE), P(FAKE), P(FAKE), P(FAKE)) == 1
    assert lib.hq_host_pipeline_wait(None) == 1
    assert lib.hq_host_pipeline_destroy(None) == 0
    assert lib.hq_host_pipeline_inject_failure(None, 1) == 1


def test_delayed_argument_checks(lib):
    def dl(x=FAKE, dt=1, M=4, K=32, ldx=32, G=16, prev=FAKE, nxt=FAKE + 64, q=FAKE, s=FAKE, sg=None):
        return lib.hq_rotate_quant_nvfp4_delayed(
            P(x) if x else None, dt, M, K, ldx, G, P(prev) if prev else None,
            P(nxt) if nxt else None, P(q) if q else None, P(s) if s else None,
            P(sg) if sg else None, None)
    assert dl(nxt=0) == 1
    assert dl(prev=0) == 1 and dl(q=0) == 1 and dl(s=0) == 1
    assert dl(prev=FAKE + 64) == 8        # the two amax pointers alias: HQ_ERR_ALIAS
    assert dl(G=32) == 5 and dl(dt=3) == 4 and dl(K=24, ldx=24) == 2
    assert dl(nxt=FAKE + 66) == 3 and dl(q=FAKE + 8) == 3


def test_int8_argument_checks(lib):
    def i8(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, q=FAKE, s=FAKE):
        return lib.hq_rotate_quant_int8(P(x) if x else None, dt, M, K, ldx, G, P(q) if q else None,
                                        P(s) if s else None, None)
    assert i8(x=0) == 1 and i8(q=0) == 1 and i8(s=0) == 1
    assert i8(G=32) == 5 and i8(G=0) == 5 and i8(G=8) == 5 and i8(G=2048) == 5
    assert i8(dt=2) == 4
    assert i8(K=48, ldx=48, G=64) == 2 and i8(K=1536, ldx=1536, G=1024) == 2
    assert i8(K=36, ldx=36, G=4) == 2          # a multiple of 4 but not of 16
    assert i8(K=2 ** 41, ldx=2 ** 41, M=1, G=1024) == 2   # 2^30 warp tiles per row
    assert i8(ldx=32) == 2 and i8(M=-1) == 2
    assert i8(x=FAKE + 8) == 3 and i8(q=FAKE + 4) == 3 and i8(s=FAKE + 2) == 3
    assert i8(ldx=68) == 3                     # 136-byte bf16 row stride
    assert i8(M=2 ** 62) == 2 and i8(ldx=2 ** 62) == 2   # M*K, ldx*2 overflow int64
    assert i8(M=0) == 0


def test_mxfp4_argument_checks(lib):
    def mx(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, q=FAKE, s=FAKE):
        return lib.hq_rotate_quant_mxfp4(P(x) if x else None, dt, M, K, ldx, G, P(q) if q else None,
                                         P(s) if s else None, None)
    assert mx(x=0) == 1 and mx(q=0) == 1 and mx(s=0) == 1
    assert mx(K=48, ldx=48) == 2             # not a multiple of 32
    assert mx(G=64) == 5 and mx(dt=5) == 4
    assert mx(q=FAKE + 8) == 3 and mx(x=FAKE + 4) == 3

    def mxw(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, q=FAKE, s=FAKE, ws=FAKE + 256):
        return lib.hq_rotate_quant_mxfp4_ws(P(x) if x else None, dt, M, K, ldx, G, P(q) if q else None,
                                            P(s) if s else None, P(ws) if ws else None, None)
    assert mxw(x=0) == 1 and mxw(q=0) == 1 and mxw(s=0) == 1
    assert mxw(K=48, ldx=48) == 2 and mxw(G=64) == 5 and mxw(dt=5) == 4
    assert mxw(ws=FAKE + 2) == 3 and mxw(q=FAKE + 8) == 3
    assert mxw(M=0) == 0 and mxw(M=0, ws=0) == 0
    assert lib.hq_dequant_mxfp4(P(FAKE), P(FAKE), 4, 48, 0, 0, P(FAKE), None) == 2
    assert lib.hq_dequant_mxfp4(None, P(FAKE), 4, 64, 0, 0, P(FAKE), None) == 1
    assert lib.hq_dequant_mxfp4(P(FAKE), P(FAKE), 4, 64, 0, 1, P(FAKE), None) == 5


def test_delayed_ws_argument_checks(lib):
    def dw(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, ap=FAKE, an=FAKE + 64, q=FAKE, s=FAKE, sg=None, ws=FAKE + 256):
        return lib.hq_rotate_quant_nvfp4_delayed_ws(
            P(x) if x else None, dt, M, K, ldx, G, P(ap) if ap else None, P(an) if an else None,
            P(q) if q else None, P(s) if s else None, P(sg) if sg else None, P(ws) if ws else None, None)
    assert dw(an=0) == 1 and dw(ap=0) == 1 and dw(q=0) == 1 and dw(x=0) == 1
    assert dw(an=FAKE) == 8                  # amax_prev and amax_next alias
    assert dw(G=32) == 5 and dw(dt=2) == 4 and dw(K=24, ldx=24) == 2
    assert dw(ws=FAKE + 2) == 3 and dw(an=FAKE + 66) == 3


def test_swizzled_argument_checks_and_size(lib):
    def sw(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, a=FAKE, q=FAKE, s=FAKE, sg=None):
        return lib.hq_rotate_quant_nvfp4_swizzled(
            P(x) if x else None, dt, M, K, ldx, G, P(a) if a else None, P(q) if q else None,
            P(s) if s else None, P(sg) if sg else None, None)
    assert sw(a=0) == 1 and sw(q=0) == 1 and sw(s=0) == 1 and sw(x=0) == 1
    assert sw(G=32) == 5 and sw(dt=2) == 4 and sw(K=24, ldx=24) == 2
    assert sw(s=FAKE + 4) == 3 and sw(s=FAKE + 16) == 3   # the swizzled scales are 32-byte aligned

    def sww(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, a=FAKE, q=FAKE, s=FAKE, sg=None, ws=FAKE + 256):
        return lib.hq_rotate_quant_nvfp4_swizzled_ws(
            P(x) if x else None, dt, M, K, ldx, G, P(a) if a else None, P(q) if q else None,
            P(s) if s else None, P(sg) if sg else None, P(ws) if ws else None, None)
    assert sww(a=0) == 1 and sww(q=0) == 1 and sww(s=0) == 1 and sww(x=0) == 1
    assert sww(G=32) == 5 and sww(dt=2) == 4 and sww(K=24, ldx=24) == 2
    assert sww(s=FAKE + 16) == 3 and sww(ws=FAKE + 2) == 3
    assert sww(M=0) == 0 and sww(M=0, ws=0) == 0
    assert sw(q=FAKE + 8) == 3 and sw(x=FAKE + 8) == 3
    assert sw(M=0) == 0
    # tiles of 128 rows x 4 scale columns, padded
    assert lib.hq_swizzled_scales_bytes(1, 16) == 128 * 4
    assert lib.hq_swizzled_scales_bytes(128, 64) == 128 * 4
    assert lib.hq_swizzled_scales_bytes(129, 64) == 256 * 4
    assert lib.hq_swizzled_scales_bytes(200, 96) == 256 * 8
    assert lib.hq_swizzled_scales_bytes(32768, 28672) == 32768 * 1792
    assert lib.hq_swizzled_scales_bytes(0, 0) == 0
    assert lib.hq_swizzled_scales_bytes(4, 24) == -1 and lib.hq_swizzled_scales_bytes(-1, 16) == -1
    assert lib.hq_swizzled_scales_bytes(2 ** 63 - 1, 16) == -1       # would overflow int64
    assert lib.hq_swizzled_scales_bytes(2 ** 40, 2 ** 30) == -1
    assert lib.hq_swizzled_scales_bytes(2 ** 40, 64) == 2 ** 40 * 4  # the largest are exact


def test_selftest_argument_check(lib):
    assert lib.hq_selftest_bounded_wait(2, None) == 2 and lib.hq_selftest_bounded_wait(-1, None) == 2


def test_binding_has_every_abi_call_under_the_same_name():
    """The Python binding mirrors include/hq.h: one function per C entry point, same name.
    The host pipeline calls are the methods of HostQuantizer; hq_last_cuda_error is carried by
    HQError."""
    import hadamard_rotation_gb300 as hq

    wrapped_elsewhere = {"hq_host_pipeline_create", "hq_host_pipeline_destroy", "hq_host_pipeline_submit",
                         "hq_host_pipeline_wait", "hq_host_pipeline_workspace_bytes",
                         "hq_host_pipeline_inject_failure", "hq_last_cuda_error"}
    missing = [n for n in declared_functions() if n not in wrapped_elsewhere and not callable(getattr(hq, n, None))]
    assert not missing, missing
    assert hq.hq_version() == 100
    assert hq.hq_status_string(0).startswith("HQ_OK")


def test_quantize_argument_checks(lib):
    def qz(x=FAKE, dt=1, M=4, K=64, ldx=64, G=16, a=FAKE, q=FAKE, s=FAKE, sg=None, ws=FAKE + 256):
        return lib.hq_quantize_nvfp4(
            P(x) if x else None, dt, M, K, ldx, G, P(a) if a else None, P(q) if q else None,
            P(s) if s else None, P(sg) if sg else None, P(ws) if ws else None, None)
    assert qz(x=0) == 1 and qz(a=0) == 1 and qz(q=0) == 1 and qz(s=0) == 1
    assert qz(G=32) == 5 and qz(dt=2) == 4 and qz(K=24, ldx=24) == 2 and qz(M=-1) == 2
    assert qz(a=FAKE + 2) == 3 and qz(ws=FAKE + 2) == 3
    assert qz(q=FAKE + 8) == 3 and qz(s=FAKE + 2) == 3 and qz(x=FAKE + 8) == 3
    assert qz(sg=FAKE + 1) == 3
    # The two-launch cases (strided rows, x above the one-launch limit, no workspace) check
    # the outputs before pass 1 is enqueued too: without a device these would otherwise
    # report the failed launch (6).
    for kw in (dict(ldx=128), dict(M=65536, K=1024, ldx=1024), dict(ws=0)):
        assert qz(q=0, **kw) == 1 and qz(s=0, **kw) == 1
        assert qz(q=FAKE + 8, **kw) == 3 and qz(s=FAKE + 2, **kw) == 3 and qz(sg=FAKE + 1, **kw) == 3
    assert qz(M=2 ** 40, K=2 ** 22, ldx=2 ** 22, q=0) == 1   # M*K*4 would overflow int64


def test_binding_constants_match_the_header():
    from hadamard_rotation_gb300 import api

    text = open(HEADER).read()
    words = re.search(r"#define HQ_QUANTIZE_WORKSPACE_WORDS (\d+)", text)
    assert words and int(words.group(1)) == api.HQ_QUANTIZE_WORKSPACE_WORDS


def test_noalloc_argument_checks_and_size_limit(lib):
    # hq_quantize_nvfp4_host_noalloc checks its arguments and the size of its fixed device
    # array before it makes any CUDA call, so every status below is decided on the host.
    def na(x=FAKE, dt=1, M=4, K=32, G=16, q=FAKE, s=FAKE, sg=FAKE):
        return lib.hq_quantize_nvfp4_host_noalloc(
            P(x) if x else None, dt, M, K, G, P(q) if q else None, P(s) if s else None,
            P(sg) if sg else None, None)
    assert na(x=0) == 1 and na(q=0) == 1 and na(s=0) == 1 and na(sg=0) == 1
    assert na(G=32) == 5 and na(dt=2) == 4
    assert na(K=24) == 2 and na(K=272, G=256) == 2 and na(M=-1) == 2
    assert na(M=2 ** 62, K=64) == 2               # M*K overflows
    assert na(M=0, x=0) == 0                      # empty: nothing to do
    # The array holds r(n*e) + r(n/2) + r(n/16) + 512 bytes, r() rounding up to 256 bytes.
    limit = 32 * 1024 * 1024
    assert "#define HQ_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)" in open(HEADER).read()

    def need(n, e):
        r = lambda b: (b + 255) // 256 * 256
        return r(n * e) + r(n // 2) + r(n // 16) + 512

    for dt, e, rows in ((1, 2, 3196), (0, 4, 1795)):  # the most rows of 4096 that fit
        assert need(rows * 4096, e) <= limit < need((rows + 1) * 4096, e)
        assert na(dt=dt, M=rows + 1, K=4096) == 7
        if not torch.cuda.is_available():
            assert na(dt=dt, M=rows, K=4096) == 6     # fits: the call reaches the runtime
    assert na(M=2 ** 41, K=16) == 7
