"""The multi-rank host logic of bench.py on CPU (gloo, world size 2, 127.0.0.1).

bench.py --gpus N runs N independent replicas; the only exchange is host-side: a barrier and
the maximum over ranks of the timed region, from which rank 0 reports whole-job throughput.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = 10.0 + 5.0 * rank
    worst = bench.max_over_ranks(mine)
    gbs = bench.throughput_gbs(1_000_000_000, 4, world, worst)
    dist.barrier()
    q.put((rank, worst, gbs))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in results] == [15.0, 15.0]          # every rank sees the slowest time
    assert results[0][2] == pytest.approx(1e9 * 4 * 2 / 0.015 / 1e9)  # all ranks' bytes / max time


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.throughput_gbs(2_000_000_000, 10, 1, 1000.0) == pytest.approx(20.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "tiny_f32_128x256"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_traffic_table_keys_name_a_source_a_workload_and_a_group():
    # Each captured traffic figure is keyed by the kernel source hash it was taken on (16 hex
    # digits, the form kernel_source_hash() returns), a named workload and a rotation group, and
    # is no larger than the bytes a launch could move if it read every input byte and wrote
    # every output byte twice.
    sys.path.insert(0, ROOT)
    import bench
    from hadamard_rotation_gb300 import synth

    assert len(bench.kernel_source_hash()) == 16
    for (source, name, group), traffic in bench.NCU_TRAFFIC.items():
        assert len(source) == 16 and int(source, 16) >= 0
        assert name in synth.WORKLOADS and group in synth.WORKLOADS[name].groups
        w = synth.WORKLOADS[name]
        assert 0 < traffic <= 2 * (w.bytes_in() + w.bytes_out())
