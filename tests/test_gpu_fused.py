"""hq_quantize_nvfp4, both passes in one call (two launches), against the CPU oracle.

With a workspace, pass 1 reduces the amax into it (no memset) and pass 2 takes its tiles from the
workspace's counters (from 16384 warp tiles on) and fetches its first tiles while pass 1 ends;
without, the plain hq_rot_amax then hq_rotate_quant_nvfp4.  Either way amax, s_global, codes and
scales must be bit-exact with the oracle, and the workspace must be back to zero after every call
(the next call relies on it).  hq_rotate_quant_nvfp4_ws, pass 2 with the run-time split, is
tested here too.
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


# A finished call leaves every workspace word 0 (the next call relies on it).
def settled(ws) -> bool:
    return not ws.any().item()


def f32_bits(a) -> np.ndarray:
    return np.asarray(a, np.float32).view(np.uint32)


def rand_input(M, K, dtype, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32) * np.float32(scale)
    if K >= 64:
        cols = rng.choice(K, max(1, K // 64), replace=False)
        x[:, cols] *= 30.0
    if M > 3:
        x[2] = 0.0
    t = torch.from_numpy(x)
    return t if dtype == torch.float32 else t.to(dtype)


def check(x_host, group, got, label):
    q, s, sg, amax = (t.cpu().numpy() for t in got)
    oq, os_, oamax, osg = oracle.quantize(synth.as_oracle_array(x_host), group)
    assert f32_bits(amax)[0] == f32_bits([oamax])[0], (label, amax, oamax)
    assert f32_bits(sg)[0] == f32_bits([osg])[0], (label, sg, osg)
    for name, a, b in (("scales", s, os_), ("codes", q, oq)):
        if not np.array_equal(a, b):
            idx = np.argwhere(a != b)[:5]
            raise AssertionError(f"{label} {name}: {int(np.count_nonzero(a != b))} differ, first {idx.tolist()}")


def kernels_launched(fn):
    """Names of the CUDA kernels `fn` launches (torch's profiler); None if it sees none."""
    from torch.profiler import ProfilerActivity, profile

    with profile(activities=[ProfilerActivity.CUDA]):  # the first session can miss events
        torch.ones(1, device="cuda").add_(1)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = [e.name for e in prof.events() if e.device_type == torch.autograd.DeviceType.CUDA]
    return names or None


SHAPES = [(1, 256), (2, 16 * 16), (129, 256), (77, 4096), (1000, 1024), (4099, 512)]


@pytest.mark.parametrize("M,K", SHAPES)
@pytest.mark.parametrize("group", [0, 16, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_matches_oracle(M, K, group, dtype):
    x_host = rand_input(M, K, dtype, seed=M * 3 + K + group)
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    got = hq.hq_quantize_nvfp4(x_host.cuda(), group, workspace=ws)
    torch.cuda.synchronize()
    check(x_host, group, got, f"{M}x{K} {dtype}")
    assert settled(ws), ws


@pytest.mark.parametrize("group", [0, 16, 256])
def test_named_4096x4096_workload(group):
    w = synth.WORKLOADS["bf16_4096x4096"]
    x_host = synth.generate(w)
    x = x_host.cuda()
    got = hq.quantize_nvfp4(x, group)
    torch.cuda.synchronize()
    check(x_host, group, got, f"bf16 [4096, 4096] group {group}")
    names = kernels_launched(lambda: hq.quantize_nvfp4(x, group))
    if names is None:
        pytest.skip("the profiler sees no CUDA kernels here")
    assert len(names) == 2 and "k_rot_amax" in names[0] and "k_rotate_quant_nvfp4" in names[1], names


def test_repeated_calls_reuse_the_workspace():
    """A large-amax tensor, then a small-amax one, then the first again, with one workspace:
    each amax is exact, so the accumulator and the CTA count were reset in between."""
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    xs = [rand_input(300, 2048, torch.bfloat16, seed=5, scale=100.0),
          rand_input(300, 2048, torch.bfloat16, seed=6, scale=0.01),
          rand_input(300, 2048, torch.bfloat16, seed=5, scale=100.0)]
    for i, x_host in enumerate(xs):
        for group in (16, 256):
            got = hq.hq_quantize_nvfp4(x_host.cuda(), group, workspace=ws)
            torch.cuda.synchronize()
            check(x_host, group, got, f"call {i} group {group}")
            assert settled(ws)


def test_two_launches_with_a_workspace_leave_it_zero():
    """Strided rows always take the two launches; with a workspace, pass 1 reduces the amax
    into it (no memset before the launch) and its last CTA writes amax.  A large, a small and
    a large amax in turn, every group and both input types (the streaming pass 1 needs
    contiguous rows, so the tiled one runs here; the next test covers the streaming one): every
    result exact and the workspace back to 0 after each call."""
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    for dtype in (torch.bfloat16, torch.float32):
        for i, scale in enumerate((100.0, 0.01, 100.0)):
            x_host = rand_input(300, 2048, dtype, seed=40 + i, scale=scale)
            padded = torch.zeros(300, 2048 + 256, dtype=dtype, device="cuda")
            padded[:, :2048] = x_host.cuda()
            for group in (0, 16, 256):
                got = hq.hq_quantize_nvfp4(padded[:, :2048], group, workspace=ws)
                torch.cuda.synchronize()
                check(x_host, group, got, f"strided {dtype} call {i} group {group}")
                assert settled(ws)


def test_streaming_pass_1_with_a_workspace_in_a_row():
    """Contiguous bf16 rows: the streaming pass 1 reduces into the workspace, and pass 2 (16400
    warp tiles) takes the run-time split.  Two different tensors in a row on one workspace, both
    exact, workspace 0."""
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    for seed, scale in ((51, 7.0), (52, 0.003)):
        x_host = rand_input(8200, 4096, torch.bfloat16, seed=seed, scale=scale)
        got = hq.hq_quantize_nvfp4(x_host.cuda(), 16, workspace=ws)
        torch.cuda.synchronize()
        check(x_host, 16, got, f"bf16 [8200, 4096] seed {seed}")
        assert settled(ws)


def test_two_launch_modes_agree():
    """Without a workspace (hq_rot_amax then hq_rotate_quant_nvfp4) and on strided rows (the
    fixed split) the bytes are those of the workspace path."""
    x_host = rand_input(640, 3072, torch.bfloat16, seed=17)
    x = x_host.cuda()
    a = hq.hq_quantize_nvfp4(x, 16)
    b = hq.hq_quantize_nvfp4(x, 16, use_workspace=False)
    big = torch.zeros(640, 3072 + 256, dtype=torch.bfloat16, device="cuda")
    big[:, :3072] = x
    c = hq.hq_quantize_nvfp4(big[:, :3072], 16)
    torch.cuda.synchronize()
    for other in (b, c):
        for u, v in zip(a, other):
            assert torch.equal(u, v)
    check(x_host, 16, a, "640x3072")


def test_zero_empty_and_nonfinite():
    x = torch.zeros(64, 256, device="cuda")
    q, s, sg, amax = hq.quantize_nvfp4(x, 16)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and sg.item() == 1.0 and not q.any().item() and not s.any().item()
    e = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    q, s, sg, amax = hq.quantize_nvfp4(e, 16)
    torch.cuda.synchronize()
    assert amax.item() == 0.0 and q.numel() == 0
    x = torch.ones(64, 256, device="cuda")
    x[33, 7] = float("inf")
    for group in (0, 16, 256):
        assert torch.isinf(hq.quantize_nvfp4(x, group)[3]).item()
    x[12, 200] = float("nan")
    for group in (0, 16, 256):
        assert torch.isnan(hq.quantize_nvfp4(x, group)[3]).item()
    assert hq.hq_read_fault() == 0


def test_two_streams_at_once():
    """Calls on two streams, in flight together, each with the workspace the binding keeps for
    its stream."""
    xs = [rand_input(2048, 2048, torch.bfloat16, seed=40 + i) for i in range(2)]
    xd = [x.cuda() for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = [None, None]
    for _ in range(4):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs[i] = hq.quantize_nvfp4(xd[i], 16, stream=streams[i])
    torch.cuda.synchronize()
    for i in range(2):
        check(xs[i], 16, outs[i], f"stream {i}")


@pytest.mark.parametrize("use_ws", [True, False])
def test_cuda_graph_capture_and_replay(use_ws):
    """Both paths captured in a CUDA graph and replayed on new contents of the same input
    buffer: every replay is exact (the workspace, whose pass 2 takes the run-time split on this
    tensor of 16384 warp tiles, is zero again after each)."""
    xs = [rand_input(4096, 8192, torch.bfloat16, seed=70 + i, scale=10.0 ** (i - 1)) for i in range(3)]
    x = xs[0].cuda()
    amax = torch.empty(1, device="cuda")
    q = torch.empty((4096, 4096), dtype=torch.uint8, device="cuda")
    s = torch.empty((4096, 512), dtype=torch.uint8, device="cuda")
    sg = torch.empty(1, device="cuda")
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture (grid sizes, attributes)
        hq.hq_quantize_nvfp4(x, 16, amax=amax, q=q, scales=s, s_global=sg, use_workspace=use_ws,
                             workspace=ws if use_ws else None, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        hq.hq_quantize_nvfp4(x, 16, amax=amax, q=q, scales=s, s_global=sg, use_workspace=use_ws,
                             workspace=ws if use_ws else None)
    for i, x_host in enumerate(xs):
        x.copy_(x_host.cuda())
        g.replay()
        torch.cuda.synchronize()
        check(x_host, 16, (q, s, sg, amax), f"replay {i} workspace={use_ws}")
        assert settled(ws)


@pytest.mark.parametrize("M,K", [(1, 16), (999, 4352), (4099, 8192), (16385, 2048), (2053, 17408)])
def test_pass_2_with_run_time_tile_schedule(M, K):
    """hq_rotate_quant_nvfp4_ws hands the tiles out from counters in the workspace from 16384
    warp tiles on (below, and for strided rows, it is the fixed split).  Small sizes (one
    block; fewer tiles than warps) and sizes past the threshold with a ragged last tile (16385
    x 2048: 16385 tiles, 2053 x 17408: 17449 tiles, classes of unequal length); contiguous and
    strided rows, both input types, every group it can take; each call twice in a row on one
    workspace.  Codes, scales and s_global equal the oracle's, and the workspace is 0 after
    every call."""
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
    for dtype in (torch.bfloat16, torch.float32):
        x_host = rand_input(M, K, dtype, seed=M + K)
        xo = synth.as_oracle_array(x_host)
        for strided in (False, True):
            if strided:
                xd = torch.zeros(M, K + 64, dtype=dtype, device="cuda")
                xd[:, :K] = x_host.cuda()
                x = xd[:, :K]
            else:
                x = x_host.cuda()
            for group in (0, 16, 256):
                if K % max(group, 16):
                    continue
                oq, os_, oamax, osg = oracle.quantize(xo, group)
                amax = torch.tensor([oamax], dtype=torch.float32, device="cuda")
                label = f"{dtype} [{M}, {K}] strided={strided} group={group}"
                for call in range(2):
                    q, s, sg = hq.hq_rotate_quant_nvfp4_ws(x, group, amax, workspace=ws)
                    torch.cuda.synchronize()
                    assert f32_bits(sg.cpu().numpy())[0] == f32_bits([osg])[0], label
                    assert np.array_equal(s.cpu().numpy(), os_), (label, call)
                    assert np.array_equal(q.cpu().numpy(), oq), (label, call)
                    assert settled(ws), (label, call)
    assert hq.hq_read_fault() == 0


def test_run_time_schedule_on_two_streams_with_their_own_workspaces():
    """Two streams quantize two tensors at the same time, each with its own workspace (the
    documented rule for calls that may overlap): both results exact, both workspaces 0."""
    xs = [rand_input(4096, 8192, torch.bfloat16, seed=61 + i) for i in range(2)]  # 16384 tiles
    streams = [torch.cuda.Stream() for _ in xs]
    wss = [torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
           for _ in xs]
    xd = [x.cuda() for x in xs]
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):
        outs = []
        for x, st, ws in zip(xd, streams, wss):
            with torch.cuda.stream(st):
                amax = hq.hq_rot_amax(x, 16, stream=st)
                outs.append(hq.hq_rotate_quant_nvfp4_ws(x, 16, amax, workspace=ws, stream=st))
    torch.cuda.synchronize()
    for x_host, (q, s, sg), ws in zip(xs, outs, wss):
        oq, os_, _, osg = oracle.quantize(synth.as_oracle_array(x_host), 16)
        assert np.array_equal(q.cpu().numpy(), oq) and np.array_equal(s.cpu().numpy(), os_)
        assert settled(ws)


def test_workspace_forms_on_two_streams_with_their_own_workspaces():
    """The swizzled-scale pass (units handed out at run time), MXFP4 and the delayed pass (tiles
    handed out at run time) on two streams at the same time, each stream with its own
    workspace, three rounds: every result exact, every workspace 0."""
    xs = [rand_input(4099, 8192, torch.bfloat16, seed=71 + i) for i in range(2)]
    streams = [torch.cuda.Stream() for _ in xs]
    wss = [torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device="cuda")
           for _ in xs]
    xd = [x.cuda() for x in xs]
    amaxes = [hq.hq_rot_amax(x, 16) for x in xd]
    torch.cuda.synchronize()
    for _ in range(3):
        outs = []
        for x, st, ws, amax in zip(xd, streams, wss, amaxes):
            with torch.cuda.stream(st):
                sw = hq.hq_rotate_quant_nvfp4_swizzled_ws(x, 16, amax, workspace=ws, stream=st)
                mx = hq.hq_rotate_quant_mxfp4_ws(x, 16, workspace=ws, stream=st)
                dl = hq.hq_rotate_quant_nvfp4_delayed_ws(x, 16, amax, workspace=ws, stream=st)
                outs.append((sw, mx, dl))
        torch.cuda.synchronize()
        for x_host, (sw, mx, dl), ws in zip(xs, outs, wss):
            xo = synth.as_oracle_array(x_host)
            oq, os_, oamax, osg = oracle.quantize(xo, 16)
            assert np.array_equal(sw[0].cpu().numpy(), oq)
            assert np.array_equal(sw[1].cpu().numpy(), oracle.swizzle_scales(os_))
            mq, ms = oracle.quantize_mxfp4(xo, 16)
            assert np.array_equal(mx[0].cpu().numpy(), mq) and np.array_equal(mx[1].cpu().numpy(), ms)
            assert np.array_equal(dl[0].cpu().numpy(), oq) and np.array_equal(dl[1].cpu().numpy(), os_)
            assert f32_bits(dl[3].cpu().numpy())[0] == f32_bits([oamax])[0]
            assert settled(ws)
