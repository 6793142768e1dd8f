"""Benchmark: fused Hadamard rotation + NVFP4 quantization on GB300.

One step = the whole hot path over one activation tensor already resident in HBM, as
hq_quantize_nvfp4 runs it with a workspace: pass 1 (rotate, global amax, reduced into the
workspace) then pass 2 (rotate, block scales, codes; tiles handed out at run time), two
launches chained by programmatic dependent launch.  The metric is GB/s of algorithmic bytes
in + out per step:
    bytes = M*K*sizeof(x)  (x read)  +  M*K/2 (codes)  +  M*K/16 (E4M3 scales).
Default workload: x bf16 [32768, 28672] (1.88 GB, larger than L2, so no flush is needed
between steps), N(0,1) with 0.5% outlier channels x100, seed 3, rotation group 16.

Also reported on the same JSON line:
  roofline      the dominant kernel (pass 2): its algorithmic bytes / its average launch time
                (CUDA events around every launch in an instrumented run of the step), against
                the measured HBM copy bandwidth;
  e2e           the same metric through the public API with host buffers: pinned host x ->
                device, both passes, codes + scales + s_global -> pinned host, every step;
  cpu_baseline  the CPU oracle on a bounded sample of the workload, on this host's cores;
  clocks        nvidia-smi samples taken during the timed region.

--impl reference times the CPU oracle (the definition the kernels are checked against) as the
reference arm; it uses no GPU.

Multi-GPU: --gpus N under torchrun runs N independent replicas (one tensor per GPU, weak
scaling, no collective on the data path); the barrier and max-over-ranks time are host-side.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "bf16_32768x28672"
METRIC = "rotate+NVFP4-quant GB/s (bytes in+out) and % of GB300 HBM peak"
L2_BYTES = 126 * 1024 * 1024

# DRAM traffic per launch of the dominant kernel from a one-pass ncu capture of the bench
# workload itself (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the kernel source
# it was taken on: a changed kernel reports null until it is captured again.
NCU_TRAFFIC = {
    ("4f20776c7d3b556d", "bf16_32768x28672", 16): 1879127040 + 495954176,
}


def _code_only(text: str) -> str:
    """Source text without comments and blank space, so that only code changes move the hash
    (C/C++ // and /* */ comments; Python # comments and docstrings are kept as they are)."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the kernels' code (comments excluded), the launch code and the build script."""
    h = hashlib.sha256()
    for rel in ("hadamard_rotation_gb300/csrc/hq_kernels.cuh", "hadamard_rotation_gb300/csrc/hq.cu",
                "hadamard_rotation_gb300/build.py"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        h.update((_code_only(text) if rel.endswith((".cuh", ".cu")) else text).encode())
    return h.hexdigest()[:16]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--group", type=int, default=None, help="rotation group (default: the workload's first)")
    ap.add_argument("--e2e-steps", type=int, default=None, help="steps of the host-buffer run (default: min(steps, 200))")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload measurements reported under 'configs'")
    ap.add_argument("--rows", type=int, default=None,
                    help="only the first ROWS rows of the workload (same K, distribution and "
                         "seed): small cases of the same row shape for profiling; not a metric line")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def max_over_ranks(value_ms: float) -> float:
    """The largest of every rank's value (a host-side gloo all-reduce); the value itself when
    no process group is initialised."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value_ms)
    t = torch.tensor([float(value_ms)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput_gbs(bytes_per_step_per_rank: int, steps: int, world: int, region_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed divided by the slowest rank's time."""
    return bytes_per_step_per_rank * steps * world / (region_ms / 1e3) / 1e9


def time_launches(fn, K: int, stream, dev, flush) -> float:
    """Average milliseconds of one call of fn over K calls (CUDA events on the launching
    stream, 3 untimed calls first).  Without a flush the calls run back to back between two
    events; with one, the L2 flush runs between calls and each call has its own event pair,
    so the flush is not timed."""
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize(dev)
    if flush is None:
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / K
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        flush.fill_(1.0)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / K


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------------- clocks ------

class ClockSampler:
    """nvidia-smi samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and not (parts[1].endswith(self.uuid) or self.uuid.endswith(parts[1])):
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        pw = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def device_uuid(dev) -> str | None:
    import torch

    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u.replace("GPU-", "")
    except Exception:
        return None


# --------------------------------------------------------------------- CPU oracle ------

def oracle_sample_run(w, rows: int, reps: int, warm: int = 1, threads: int | None = None):
    """Time the CPU oracle (both passes) on the first `rows` rows of the workload, on `threads`
    threads (default: every core)."""
    import oracle
    from hadamard_rotation_gb300 import synth

    oracle.build()
    x = synth.as_oracle_array(synth.generate(w, rows=slice(0, rows)))
    group = w.groups[0]
    threads = threads or os.cpu_count() or 1
    for _ in range(warm):
        oracle.quantize(x, group, nthreads=threads)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.quantize(x, group, nthreads=threads)
        times.append(time.perf_counter() - t0)
    nbytes = rows * w.K * w.elem_bytes + rows * w.K // 2 + rows * w.K // 16
    return nbytes, times, threads


def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0  # the reference arm runs on rank 0 only; other ranks exit without work
    # Size the per-step sample so the whole run (warm-up + steps) takes about two minutes:
    # calibrate the oracle's rate on 64 rows first.
    _, t_cal, _ = oracle_sample_run(w, min(w.M, 64), reps=1, warm=1)
    per_row = max(t_cal[0] / min(w.M, 64), 1e-7)
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(min(w.M, max(1, budget / per_row)))
    nbytes, times, threads = oracle_sample_run(w, rows, reps=args.steps, warm=args.warmup)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = f"rows 0..{rows - 1} of {w.name} ({rows}x{w.K}), both passes per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / len(times) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.describe(), "group": w.groups[0], "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------- GPU arm -----

def graph_ms_per_call(fn, calls: int, reps: int, dev) -> float:
    """Median milliseconds per call of fn, from `reps` replays of a CUDA graph that holds
    `calls` calls in a row (captured once; the replays have no host work between launches, so
    short kernels are not starved by the Python binding's per-call cost)."""
    import torch

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):  # warm-up outside the capture (grid sizes, attributes)
        for _ in range(3):
            fn()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b) / calls)
    del g
    return statistics.median(times)


def measure_configs(hq, synth, dev, stream, peak: float, have: dict, launches: int = 100,
                    reps: int = 5) -> dict:
    """Every named workload and rotation mode, timed the same way: pass 2 alone (as the step
    runs it, hq_rotate_quant_nvfp4_ws), pass 1 alone (hq_rot_amax) and the whole step
    (hq_quantize_nvfp4 with a workspace), each as `launches` calls back to back in one CUDA
    graph, median of `reps` replays timed by CUDA events.

    Inputs larger than L2 are read from HBM by construction.  For an input that L2 holds, the
    calls cycle through enough copies of x and of the outputs that each call reads an x last
    touched at least three L2 capacities earlier; the same calls are also timed cold, one call
    per event pair after an L2 flush (the flush outside the pair), which adds the launch
    latency to every figure.  `have` maps workload names to device tensors already made."""
    import torch

    out = {}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    for name in synth.WORKLOAD_ORDER:
        w = synth.WORKLOADS[name]
        x0 = have.get(name)
        if x0 is None:
            x0 = synth.generate(w).to(dev)
        bin_, bout = w.bytes_in(), w.bytes_out()
        nb = bin_ + bout
        small = nb < 2 * L2_BYTES
        copies = 1
        if small and nb >= (8 << 20):
            copies = min(64, -(-3 * L2_BYTES // nb) + 1)
        xs = [x0] + [x0.clone() for _ in range(copies - 1)]
        qs = [torch.empty((w.M, w.K // 2), dtype=torch.uint8, device=dev) for _ in range(copies)]
        ss = [torch.empty((w.M, w.K // 16), dtype=torch.uint8, device=dev) for _ in range(copies)]
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        a1 = torch.empty(1, dtype=torch.float32, device=dev)
        sg = torch.empty(1, dtype=torch.float32, device=dev)
        ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)
        ws2 = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)
        entry = {"workload": w.describe(), "M": w.M, "K": w.K, "input_dtype": w.dtype,
                 "bytes_per_step": nb,
                 "timing": ("inputs larger than L2; calls back to back in a CUDA graph" if not small else
                            (f"calls back to back in a CUDA graph over {copies} copies of x and the "
                             f"outputs ({copies * nb / 1e6:.0f} MB), no flush; cold: L2 flushed "
                             "before each call, one event pair per call" if copies > 1 else
                             "cold only: L2 flushed before each call, one event pair per call")),
                 "groups": {}}
        for group in w.groups:
            hq.hq_rot_amax(x0, group, amax=amax, stream=stream)
            i = [0]

            def nxt():
                k = i[0] % copies
                i[0] += 1
                return k

            # the calls take the current stream, so that a graph capture records them
            def p2():  # pass 2 as the step runs it (run-time tile split from 16384 tiles on)
                k = nxt()
                hq.hq_rotate_quant_nvfp4_ws(xs[k], group, amax, q=qs[k], scales=ss[k], s_global=sg,
                                            workspace=ws2)

            def p1():
                hq.hq_rot_amax(xs[nxt()], group, amax=a1)

            def st():
                k = nxt()
                hq.hq_quantize_nvfp4(xs[k], group, amax=a1, q=qs[k], scales=ss[k], s_global=sg,
                                     workspace=ws)

            g = {}
            for key, fn in (("pass2", p2), ("pass1", p1), ("step", st)):
                if copies > 1 or not small:
                    i[0] = 0
                    g[f"{key}_ms"] = graph_ms_per_call(fn, launches, reps, dev)
                if small:
                    g[f"{key}_cold_ms"] = time_launches(fn, 50, torch.cuda.current_stream(dev), dev, flush)
            for suffix in ("", "_cold"):
                if f"pass2{suffix}_ms" not in g:
                    continue
                p2ms, p1ms, stms = (g[f"pass2{suffix}_ms"], g[f"pass1{suffix}_ms"], g[f"step{suffix}_ms"])
                g[f"pass2{suffix}_gbs"] = nb / (p2ms / 1e3) / 1e9
                g[f"pass2{suffix}_frac_of_peak"] = g[f"pass2{suffix}_gbs"] / peak
                g[f"pass2{suffix}_frac_of_nominal_8000"] = g[f"pass2{suffix}_gbs"] / 8000.0
                g[f"pass1{suffix}_gbs_read"] = bin_ / (p1ms / 1e3) / 1e9
                g[f"step{suffix}_gbs"] = nb / (stms / 1e3) / 1e9
                g[f"step{suffix}_gbs_both_reads"] = (2 * bin_ + bout) / (stms / 1e3) / 1e9
            g["step_path"] = "pass 1 then pass 2, two launches"
            entry["groups"]["off" if group == 0 else str(group)] = g
        out[name] = entry
        del xs, qs, ss, x0
        torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch

    import hadamard_rotation_gb300 as hq
    from hadamard_rotation_gb300 import build as hq_build
    from hadamard_rotation_gb300 import synth

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm has no CPU path)")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist

        # control plane only (barrier, max of the timings): replicas exchange no data
        dist.init_process_group("gloo")
        pg = dist
    hq_build.build()
    hq.load()
    group = args.group if args.group is not None else w.groups[0]

    x_host = synth.generate(w).pin_memory()
    x = x_host.to(dev)
    bytes_in = x.numel() * x.element_size()
    bytes_out = w.numel // 2 + w.numel // 16
    step_bytes = bytes_in + bytes_out
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    q = torch.empty((w.M, w.K // 2), dtype=torch.uint8, device=dev)
    s = torch.empty((w.M, w.K // 16), dtype=torch.uint8, device=dev)
    sg = torch.empty(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = None
    if bytes_in + bytes_out < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    # The step is one hq_quantize_nvfp4 call with a workspace: pass 1 then pass 2 as two
    # launches, pass 1 reducing into the workspace (no memset before it).
    ws = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)
    ws2 = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)

    def pass1():
        hq.hq_rot_amax(x, group, amax=amax, stream=stream)

    def pass2():  # pass 2 as the step runs it (run-time tile split from 16384 tiles on)
        hq.hq_rotate_quant_nvfp4_ws(x, group, amax, q=q, scales=s, s_global=sg, workspace=ws2,
                                    stream=stream)

    def step():
        hq.hq_quantize_nvfp4(x, group, amax=amax, q=q, scales=s, s_global=sg, workspace=ws,
                             stream=stream)

    for _ in range(args.warmup):
        step()
        if flush is not None:
            flush.fill_(1.0)
    torch.cuda.synchronize(dev)

    K = args.steps
    # The timed region holds the steps and nothing else: a CUDA event recorded between two
    # launches costs the GPU about 2 us, so per-pass events would lengthen a step (6 us per
    # step with three of them).  Without an L2 flush the region is timed by one event pair;
    # with one, each step has its own pair so that the flush between steps is not timed.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)] if flush is not None else None
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(device_uuid(dev))
    sampler.start()
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        if flush is None:
            step()
        else:
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
            flush.fill_(1.0)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if pg:
        pg.barrier()
    region_ms = t_start.elapsed_time(t_end)
    if flush is not None:
        # steps are timed launch to launch; the L2 flush between them is not part of a step
        region_ms = sum(a.elapsed_time(b) for a, b in ev)
    region_ms = max_over_ranks(region_ms)
    step_ms = region_ms / K
    value = throughput_gbs(step_bytes, K, world, region_ms)

    # ---- the passes, from a second run of the same step with an event between them ----
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        evp[i][0].record(stream)
        pass1()
        evp[i][1].record(stream)
        pass2()
        evp[i][2].record(stream)
        if flush is not None:
            flush.fill_(1.0)
    torch.cuda.synchronize(dev)
    pass1_ms = [evp[i][0].elapsed_time(evp[i][1]) for i in range(K)]
    pass2_ms = [evp[i][1].elapsed_time(evp[i][2]) for i in range(K)]
    instrumented_step_ms = sum(evp[i][0].elapsed_time(evp[i][2]) for i in range(K)) / K

    # ---- single-pass mode (delayed amax): one kernel per step, reported beside the step ----
    # each call quantizes with the amax the previous call reduced (two buffers alternate)
    amax_b = torch.empty(1, dtype=torch.float32, device=dev)
    calls = [0]

    ws_d = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)

    def delayed_call():
        src, dst = (amax, amax_b) if calls[0] % 2 == 0 else (amax_b, amax)
        calls[0] += 1
        hq.hq_rotate_quant_nvfp4_delayed_ws(x, group, src, amax_next=dst, q=q, scales=s,
                                            s_global=sg, workspace=ws_d, stream=stream)

    single_ms = time_launches(delayed_call, K, stream, dev, flush)

    # ---- pass 2 with the block scales in the swizzled GEMM layout, same tensor ----
    s_sw = torch.empty(hq.hq_swizzled_scales_bytes(w.M, w.K), dtype=torch.uint8, device=dev)
    ws_sw = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)
    sw_ms = time_launches(lambda: hq.hq_rotate_quant_nvfp4_swizzled_ws(
        x, group, amax, q=q, scales=s_sw, s_global=sg, workspace=ws_sw, stream=stream), K, stream, dev,
        flush)
    swz = {"group": group, "ms_per_launch": sw_ms, "bytes_per_launch": step_bytes,
           "gbs": step_bytes / (sw_ms / 1e3) / 1e9,
           "note": "hq_rotate_quant_nvfp4_swizzled_ws: pass 2 writing the scales in the 128x4-tile "
                   "layout of block-scaled NVFP4 GEMMs (units handed out at run time)"}
    del s_sw, ws_sw

    # ---- MXFP4 (E8M0 per 32, single pass) on the same tensor and group ----
    mx = None
    if w.K % 32 == 0:
        s_mx = torch.empty((w.M, w.K // 32), dtype=torch.uint8, device=dev)
        ws_mx = torch.zeros(hq.api.HQ_QUANTIZE_WORKSPACE_WORDS, dtype=torch.int32, device=dev)
        mx_ms = time_launches(lambda: hq.hq_rotate_quant_mxfp4_ws(x, group, q=q, scales=s_mx,
                                                                  workspace=ws_mx, stream=stream),
                              K, stream, dev, flush)
        mx_bytes = bytes_in + w.numel // 2 + w.numel // 32
        mx = {"group": group, "ms_per_launch": mx_ms, "bytes_per_launch": mx_bytes,
              "gbs": mx_bytes / (mx_ms / 1e3) / 1e9,
              "note": "hq_rotate_quant_mxfp4_ws (one pass: no global scale; tiles handed out at "
                      "run time)"}
        del s_mx, ws_mx

    # ---- INT8 per-token rotate-quant (regular Hadamard, G = 256) on the same tensor ----
    int8 = None
    if w.K <= 32768 and w.K % 256 == 0:
        q8 = torch.empty((w.M, w.K), dtype=torch.int8, device=dev)
        s8 = torch.empty(w.M, dtype=torch.float32, device=dev)
        i8_ms = time_launches(lambda: hq.hq_rotate_quant_int8(x, 256, q=q8, scales=s8, stream=stream),
                              K, stream, dev, flush)
        i8_bytes = bytes_in + w.numel + 4 * w.M
        int8 = {"group": 256, "ms_per_launch": i8_ms, "bytes_per_launch": i8_bytes,
                "gbs": i8_bytes / (i8_ms / 1e3) / 1e9,
                "note": "hq_rotate_quant_int8 (x read once, int8 codes + fp32 per-row scales)"}
        del q8, s8

    # ---- the same, on rows longer than tensor memory holds: x's bytes as rows of 65536 ----
    int8_long = None
    if w.numel % 65536 == 0:
        ml = w.numel // 65536
        xl = x.view(ml, 65536)
        q8 = torch.empty((ml, 65536), dtype=torch.int8, device=dev)
        s8 = torch.empty(ml, dtype=torch.float32, device=dev)
        il_ms = time_launches(lambda: hq.hq_rotate_quant_int8(xl, 256, q=q8, scales=s8, stream=stream),
                              K, stream, dev, flush)
        il_bytes = bytes_in + w.numel + 4 * ml
        int8_long = {"group": 256, "rows": ml, "channels": 65536, "ms_per_launch": il_ms,
                     "bytes_per_launch": il_bytes, "gbs": il_bytes / (il_ms / 1e3) / 1e9,
                     "note": "hq_rotate_quant_int8 on x viewed as [%d, 65536]: 32 warp tiles per row, "
                             "parked in tensor memory, x read once" % ml}
        del q8, s8, xl

    # ---- every named workload, the same measurement each ----
    configs = None
    if not args.no_configs:
        csampler = ClockSampler(device_uuid(dev))
        csampler.start()
        time.sleep(0.3)
        configs = measure_configs(hq, synth, dev, stream, load_peaks()[0], {w.name: x})
        configs["clocks"] = csampler.stop()

    # ---- end to end through the public API, host buffers ----
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else min(K, 200)
    del q, s  # the host pipeline holds its own device buffers
    hqz = hq.HostQuantizer(w.M, w.K, x.dtype, group, device=dev)
    for _ in range(max(3, min(args.warmup, 10))):
        hqz.submit(x_host)
    hqz.wait()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    # host clock around submissions + the final wait: every step copies x in and the
    # codes, scales and s_global out; consecutive steps overlap inside the pipeline.
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        hqz.submit(x_host)
    hqz.wait()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3)
    hqz.close()
    e2e_value = throughput_gbs(step_bytes, e2e_steps, world, e2e_ms)

    # ---- roofline of the dominant kernel (pass 2) ----
    peak, peak_kind = load_peaks()
    if int8 is not None:
        int8["frac_of_peak"] = int8["gbs"] / peak
    if int8_long is not None:
        int8_long["frac_of_peak"] = int8_long["gbs"] / peak
    if mx is not None:
        mx["frac_of_peak"] = mx["gbs"] / peak
    swz["frac_of_peak"] = swz["gbs"] / peak
    p2 = sum(pass2_ms) / len(pass2_ms)
    p1 = sum(pass1_ms) / len(pass1_ms)
    # the dominant kernel: pass 2
    dom_ms = p2
    achieved = step_bytes / (dom_ms / 1e3) / 1e9
    src_hash = kernel_source_hash()
    traffic = NCU_TRAFFIC.get((src_hash, w.name, group))
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic,
                "traffic_kernel_source": src_hash if traffic is not None else None,
                "kernel": "k_rotate_quant_nvfp4",
                "peak_source": f"{peak_kind} HBM copy (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s"}

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.describe(), "M": w.M, "K": w.K, "input_dtype": w.dtype,
                   "group": group, "bytes_per_step": step_bytes,
                   "l2": ("inputs larger than L2, no flush" if flush is None
                          else "L2 flushed between steps (256 MB write, outside the step time)"),
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "step_path": "hq_quantize_nvfp4: pass 1 then pass 2, two launches",
        "passes": {"pass1_ms": p1, "pass2_ms": p2,
                   "pass1_gbs_read": bytes_in / (p1 / 1e3) / 1e9,
                   "pass2_gbs": step_bytes / (p2 / 1e3) / 1e9,
                   "pass2_frac_of_nominal_8000": step_bytes / (p2 / 1e3) / 1e9 / 8000.0,
                   "step_gbs_both_reads": (2 * bytes_in + bytes_out) / (step_ms / 1e3) / 1e9,
                   "timed": ("a second run of the step, CUDA events before, between and after "
                             "the passes (each event adds about 2 us)"),
                   "instrumented_step_ms": instrumented_step_ms},
        "single_pass_delayed": {
            "ms_per_step": single_ms, "gbs": step_bytes / (single_ms / 1e3) / 1e9,
            "frac_of_peak": step_bytes / (single_ms / 1e3) / 1e9 / peak,
            "note": "hq_rotate_quant_nvfp4_delayed_ws: quantize with the previous step's amax while "
                    "reducing this one (one read of x, one launch); not the metric's two-pass step"},
        "swizzled_scales": swz,
        "mxfp4": mx,
        "int8_per_token": int8,
        "int8_per_token_long_rows": int8_long,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": hqz.h2d_bytes,
                "d2h_bytes_per_step": hqz.d2h_bytes, "steps": e2e_steps,
                "ms_per_step": e2e_ms / e2e_steps, "api": "HostQuantizer (hq_host_pipeline_*)",
                "timer": "host clock, wait() at the end"},
        "configs": configs,
        "gpu_launches": 2 * K,
        "clocks": clocks,
        "kernel_source": src_hash,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = min(w.M, max(1, (8192 * 28672) // w.K))
        nbytes, times, threads = oracle_sample_run(w, rows, reps=2)
        rows1 = max(1, rows // 16)
        nbytes1, times1, _ = oracle_sample_run(w, rows1, reps=2, threads=1)
        line["cpu_baseline"] = {
            "value": nbytes * len(times) / sum(times) / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of {w.name} ({rows}x{w.K}), both passes, 2 timed runs",
            "single_thread": {"value": nbytes1 * len(times1) / sum(times1) / 1e9, "unit": "GB/s",
                              "cores": 1, "sample": f"rows 0..{rows1 - 1}, both passes, 2 timed runs"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    from hadamard_rotation_gb300 import synth

    w = synth.WORKLOADS[args.workload]
    if args.rows is not None:
        if not 0 < args.rows <= w.M:
            raise SystemExit(f"--rows must be in 1..{w.M}")
        import dataclasses

        # the first rows of the named tensor: row chunks are drawn from their own seeded streams
        w = dataclasses.replace(w, name=f"{w.name}_rows{args.rows}", M=args.rows,
                                zero_rows=min(w.zero_rows, args.rows))
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
