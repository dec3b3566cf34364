#!/usr/bin/env python3
"""Throughput of fused RMSNorm + MXFP8 (rowwise + columnwise planes) on GB300.

Workload (default): x bf16 [32768, 8192], the stress recipe (rows scaled by
2^k, 1% zero blocks, 1% sub-normal blocks), gamma = 1 + 0.1 N(0, 1), eps 1e-6,
offset 0; seeded synthetic data (see mxfp8_block_scaled_rmsnorm_gb300/workloads.py).
One step = one call of ``rmsnorm_quant_mxfp8`` over the whole matrix (one
kernel launch). The metric is algorithmic HBM bytes moved per second:
read x and gamma once, write normed, both code planes and both scale planes.

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle
instead, on a bounded row sample of the same workload, on the host cores.
For N > 1 ranks (torchrun), every rank runs its own replica (weak scaling):
the path has no cross-GPU step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HBM GB/s (read+write) and % of GB300 peak, fused RMSNorm+MXFP8 quant"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fused_rmsnorm_quant_32768x8192.md")
KERNEL_SOURCES = [os.path.join(ROOT, "mxfp8_block_scaled_rmsnorm_gb300", "csrc", f)
                  for f in ("mxfp8_kernels.cu", "mx_table.h")]


def parse():
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--shape", default="32768x8192",
                   help="RxC of the stress workload (the default is the benchmark size)")
    p.add_argument("--workload", type=int, default=0, choices=[0, 1, 2, 3, 4, 5],
                   help="time seeded workload k (1-5) instead of the stress shape; the "
                        "benchmark line is workload 4, the others are side measurements")
    p.add_argument("--mm", default=None, metavar="MxNxK",
                   help="time the MXFP8 matrix multiply consumer (x quantized on the fly, "
                        "weight pre-quantized) on this problem size instead")
    p.add_argument("--planes", choices=["both", "rowwise", "columnwise"], default=None,
                   help="override the workload's MXFP8 planes (default: the workload's own)")
    p.add_argument("--update", action="store_true",
                   help="time the in-place plane update instead: both compact planes of "
                        "the workload copied into padded destination planes")
    p.add_argument("--residual", action="store_true",
                   help="time the residual variant: h = x + residual (a seeded N(0,1) matrix), "
                        "h written out, then RMSNorm + MXFP8 of h (fused workloads)")
    p.add_argument("--scale-layout", choices=["compact", "mma", "padded"], default="compact",
                   help="scale layout of the outputs (mma: tiled GEMM-operand layout; padded: "
                        "row-major with padded pitches)")
    p.add_argument("--graph", action="store_true",
                   help="capture one step in a CUDA graph and time graph replays (removes the "
                        "Python call overhead that dominates the tiny workloads)")
    p.add_argument("--vs-cublaslt", action="store_true",
                   help="with --mm: also time cuBLASLt's block-scaled MXFP8 GEMM "
                        "(torch._scaled_mm) on the same quantized operands, for comparison")
    p.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    p.add_argument("--cpu-rows", type=int, default=8192,
                   help="rows of the workload the CPU oracle is timed on")
    return p.parse_args()


def code_only(text: str) -> str:
    """C/C++/CUDA source without comments, trailing blanks and empty lines (the
    kernel sources hold no string literal with a comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def sources_sha256() -> str:
    """Hash of the kernel sources' code (comments ignored): a committed ncu
    summary stays valid across comment edits and goes stale on any code change."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(R: int, C: int):
    """dram read+write bytes per launch from the committed ncu summary, scaled
    to this launch's element count; None if absent or the kernel has changed."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith("<!-- ") and "=" in line:
            k, v = line[5:].rstrip(" ->").split("=", 1)
            fields[k.strip()] = v.strip()
    try:
        if fields.get("sources_sha256") != sources_sha256():
            return None
        per_elem = float(fields["dram_bytes_per_launch"]) / float(fields["elements"])
        return int(round(per_elem * R * C))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) taken while it runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.marks = {}

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0 = self.marks.get("load", 0) - 0.15
        t1 = self.marks.get("end", time.time()) + 0.15
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(value: float, pg, device) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if pg.get_backend() == "nccl" else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def barrier(pg, device=None):
    if pg is not None:
        if pg.get_backend() == "nccl" and device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def cpu_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    fields = {}
    try:
        for line in open("/proc/cpuinfo"):
            if ":" in line:
                k, v = (p.strip() for p in line.split(":", 1))
                fields.setdefault(k, v)
    except OSError:
        return "unknown"
    if "model name" in fields:
        return fields["model name"]
    if "CPU implementer" in fields:
        return f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def time_oracle(t, rows: int, rowwise=True, columnwise=True, threads=None):
    """Wall time of the oracle's fused map on the first ``rows`` rows, on
    ``threads`` host threads (all cores of this process by default)."""
    import numpy as np
    import oracle
    x = np.ascontiguousarray(t.x[:rows])
    t0 = time.perf_counter()
    oracle.rmsnorm_quant_mxfp8(x, t.gamma, t.eps, t.offset, rowwise, columnwise,
                               threads=threads or cpu_cores())
    return time.perf_counter() - t0


L2_BYTES = 129e6          # GB300 L2
FLUSH_BYTES = 256 << 20   # written between timed launches when the inputs fit in L2


class L2Flush:
    """Evicts earlier data from L2 before a timed launch: writes a 256 MB buffer,
    then reads another 256 MB one, so that L2 holds only clean lines of neither
    the inputs nor the outputs (a write alone would leave up to 129 MB of dirty
    lines for the timed kernel to write back)."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self, stream):
        import torch
        with torch.cuda.stream(stream):
            self.w.zero_()
            self.r.max()


def fits_l2(wl) -> bool:
    return sum(t.x.size for t in wl.tensors) * 2 <= L2_BYTES


def l2_note(wl) -> str:
    mb = sum(t.x.size for t in wl.tensors) * 2 / 1e6
    if not fits_l2(wl):
        return "inputs larger than L2 (x is %.0f MB, L2 is 129 MB); no flush" % mb
    return ("inputs fit in L2 (x is %.1f MB): before every timed launch, outside its "
            "events, a 256 MB memset and a 256 MB read on the stream flush L2 (leaving it "
            "clean); value from the summed launch times" % mb)


def load_workload(args):
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
    if args.workload:
        wl = W.config(args.workload)
    else:
        R, C = (int(v) for v in args.shape.lower().split("x"))
        wl = W.stress(R, C)
    if getattr(args, "planes", None):
        wl.rowwise = args.planes in ("both", "rowwise")
        wl.columnwise = args.planes in ("both", "columnwise")
        for tag in ("-both-", "-rowwise-"):
            if tag in wl.name:
                wl.name = wl.name.replace(tag, f"-{args.planes}-")
                break
    R, C = wl.tensors[0].shape
    return wl, R, C


def base_record(args, wl, R, C, world):
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W  # noqa: F401
    return {
        "metric": METRIC,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": wl.name,
            "tensors": len(wl.tensors),
            "rows": R, "cols": C,
            "planes": "+".join(p for p, on in (("rowwise", wl.rowwise),
                                               ("columnwise", wl.columnwise)) if on),
            "io": ("bf16 x,gamma -> bf16 normed, " if wl.fused else "bf16 w -> ")
                  + "e4m3 q_row/q_col, e8m0 s_row/s_col",
            "eps": wl.tensors[0].eps if wl.fused else None,
            "weight_offset": wl.tensors[0].offset if wl.fused else None,
            "seed": (args.workload - 1) if args.workload else 3,
            "input_sha256": wl.sha256(),
            "algorithmic_bytes_per_step": wl.algorithmic_bytes() + (
                sum(4 * t.x.size for t in wl.tensors) if getattr(args, "residual", False) else 0),
            "l2": l2_note(wl),
            "parallelism": f"replicas x{world}",
            "launch": "cuda-graph replay" if getattr(args, "graph", False) else "eager",
            "scale_layout": getattr(args, "scale_layout", "compact"),
            "residual": bool(getattr(args, "residual", False)),
            "op": ("update_planes" if getattr(args, "update", False)
                   else "add_rmsnorm_quant_mxfp8" if getattr(args, "residual", False)
                   else "rmsnorm_quant_mxfp8" if wl.fused else "quant_mxfp8"),
        },
    }


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
    wl, R, C = load_workload(args)
    if not wl.fused or len(wl.tensors) != 1:
        print(json.dumps({"impl": "reference", "unavailable":
                          "the oracle arm times the single-tensor fused workloads only"}))
        return 0
    t = wl.tensors[0]
    # bounded sample per step: calibrate on 32 rows, then size the sample so
    # that warm-up + timed steps take about a minute of wall time in total
    # (at most cpu_rows / 2 rows a step, at least one 32-row block)
    t32 = time_oracle(t, min(R, 32), wl.rowwise, wl.columnwise)
    budget = 60.0 / max(1, args.steps + args.warmup)
    fit = int(budget / max(t32, 1e-6)) * 32
    rows = min(R, max(32, min(args.cpu_rows // 2, fit) // 32 * 32))
    sample_bytes = W.algorithmic_bytes(rows, C, True, wl.rowwise, wl.columnwise)
    for _ in range(args.warmup):
        time_oracle(t, rows, wl.rowwise, wl.columnwise)
    times = [time_oracle(t, rows, wl.rowwise, wl.columnwise) for _ in range(args.steps)]
    per_step = sum(times) / len(times)
    value = sample_bytes / per_step / 1e9
    rec = base_record(args, wl, R, C, world)
    sample = (f"rows 0-{rows - 1} of {R} ({100.0 * rows / R:.1f}% of the workload), all "
              f"{C} columns, fused both planes, per step")
    rec.update({
        "impl": "reference",
        "value": value,
        "ms_per_step": per_step * 1e3,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model(),
                         "arch": platform.machine()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    })
    print(json.dumps(rec), flush=True)
    return 0


def run_mm(args, world, rank, local, pg):
    """Side measurement: TFLOP/s of mm_mxfp8 (quantize + block-scaled GEMM).

    The line's value is the whole mm_mxfp8 step (activation quantize + GEMM),
    timed after 0.4 s of continuous load, when a 1.4 kW part runs at its
    power cap. The roofline is the GEMM kernel alone (mm_mxfp8_quantized on
    the activation quantized once), timed twice: right after a short warm-up
    ("burst") and after the load. Its bound is the shape's: the tensor cores
    (against 2 x the measured bf16 burst and sustained figures), or HBM
    (against the measured copy) where moving the operands once takes longer
    than the flops at peak, as for decode-sized M."""
    import numpy as np
    import torch
    import mxfp8_block_scaled_rmsnorm_gb300 as mx
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W
    M, N, K = (int(v) for v in args.mm.lower().split("x"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    rng = np.random.default_rng(7)
    x = torch.from_numpy(W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
                         .view(np.int16)).view(torch.bfloat16).to(device)
    w = torch.from_numpy(W.to_bf16_bits(0.02 * rng.standard_normal((N, K), dtype=np.float32))
                         .view(np.int16)).view(torch.bfloat16).to(device)
    wq = mx.quantize_weight_for_mm(w)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    ws = torch.empty(mx.mm_mxfp8_workspace_size(M, K), dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    step = lambda: mx.mm_mxfp8(x, wq.q_row, wq.s_row, out=out, workspace=ws, stream=stream)
    xq = mx.quant_mxfp8(x, True, False, scale_layout="mma", stream=stream)
    gemm = lambda: mx.mm_mxfp8_quantized(xq.q_row, xq.s_row, wq.q_row, wq.s_row, out=out,
                                         stream=stream)
    # operands that fit in L2 are flushed from it before every timed launch
    in_bytes = M * K * 2 + wq.q_row.numel() + wq.s_row.numel()
    flush = L2Flush(device) if in_bytes <= L2_BYTES else None

    def timed(fn):
        """ms per call of fn over args.steps timed calls (events on the stream)."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(pg, device)
        torch.cuda.synchronize(device)
        for i in range(args.steps):
            if flush is not None:
                flush(stream)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        if flush is not None:
            total = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
        else:
            total = starts[0].elapsed_time(ends[-1])
        return max_over_ranks(total, pg, device) / args.steps

    clocks = ClockSampler(device.index)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
        gemm()
    torch.cuda.synchronize(device)
    burst_ms = timed(gemm)
    # load the GPU long enough for its power cap and the clock sampler (untimed)
    clocks.mark("load")
    t_settle = time.time() + 0.4
    while time.time() < t_settle:
        for _ in range(10):
            step()
        torch.cuda.synchronize(device)
    ms = timed(step)
    gemm_ms = timed(gemm)
    clocks.mark("end")
    clk = clocks.stop()

    def replay_us(fn, calls=20, reps=5):
        """µs per call of fn(stream) from replays of a CUDA graph of `calls`
        calls (back to back: operands that fit stay partly in L2)."""
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=side):
                for _ in range(calls):
                    fn(side)
        stream.wait_stream(side)
        graph.replay()
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / (reps * calls)

    extra = {}
    if args.graph:
        extra["gemm_graph_replay_us"] = replay_us(
            lambda st: mx.mm_mxfp8_quantized(xq.q_row, xq.s_row, wq.q_row, wq.s_row, out=out,
                                             stream=st))
    if args.vs_cublaslt:
        e8 = torch.float8_e8m0fnu

        def cub(st=None):
            with torch.cuda.stream(st if st is not None else stream):
                return torch._scaled_mm(xq.q_row.view(torch.float8_e4m3fn),
                                        wq.q_row.view(torch.float8_e4m3fn).t(),
                                        xq.s_row.view(e8), wq.s_row.view(e8),
                                        out_dtype=torch.bfloat16)
        for _ in range(3):
            cub()
        extra["cublaslt"] = {"kernel": "torch._scaled_mm (cuBLASLt block-scaled MXFP8) on the "
                                       "same quantized operands and tiled scales",
                             "avg_launch_us": timed(cub) * 1e3}
        if args.graph:
            extra["cublaslt"]["graph_replay_us"] = replay_us(cub)
    status = mx.device_status()
    if status != 0:
        raise SystemExit(f"the GEMM reported device status {status:#x}")
    flops = 2.0 * M * N * K
    tf = lambda t: flops / (t * 1e-3) / 1e12
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        bf16, bf16_sus = float(peaks["bf16_tflops"]), float(peaks["bf16_tflops_sustained"])
        src = "measured"
    except Exception:
        bf16, bf16_sus, src = 1900.0, 1700.0, "fallback"
    hbm, hbm_src = measured_peak()
    # the GEMM's algorithmic bytes: both operands' codes and scales read once,
    # the bf16 output written once
    gemm_bytes = float((N + M) * K + (N + M) * (K // 32) + 2 * M * N)
    # the roofline that bounds the shape: a decode-sized M leaves the tensor
    # cores idle behind the weight's stream from HBM
    if gemm_bytes / (hbm * 1e9) > flops / (2 * bf16 * 1e12):
        gbs = lambda t: gemm_bytes / (t * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "mxfp8_gemm_skinny_kernel (mm_mxfp8_quantized)"
                if M <= 128 else "mxfp8_gemm_kernel (mm_mxfp8_quantized)",
                "achieved": gbs(gemm_ms), "peak": hbm, "unit": "GB/s",
                "frac": gbs(gemm_ms) / hbm, "avg_launch_us": gemm_ms * 1e3,
                "bytes_per_launch": gemm_bytes,
                "peak_source": f"{hbm_src} hbm_gbs (copy)",
                "burst": {"achieved": gbs(burst_ms), "frac": gbs(burst_ms) / hbm,
                          "avg_launch_us": burst_ms * 1e3},
                "tensor_frac": tf(gemm_ms) / (2 * bf16_sus), "traffic": None}
    else:
        roof = {"bound": "tensor", "kernel": "mxfp8_gemm_kernel (mm_mxfp8_quantized)",
                "achieved": tf(gemm_ms), "peak": 2 * bf16_sus, "unit": "TFLOP/s",
                "frac": tf(gemm_ms) / (2 * bf16_sus), "avg_launch_us": gemm_ms * 1e3,
                "peak_source": f"{src} sustained bf16 x 2 (nominal fp8/bf16 ratio): "
                               "timed after 0.4 s of load",
                "burst": {"achieved": tf(burst_ms), "peak": 2 * bf16,
                          "frac": tf(burst_ms) / (2 * bf16),
                          "avg_launch_us": burst_ms * 1e3,
                          "peak_source": f"{src} burst bf16 x 2: timed right after "
                                         "a short warm-up"},
                "traffic": None}
    if rank == 0:
        print(json.dumps({
            "metric": "TFLOP/s of mm_mxfp8 (on-the-fly activation quantize + block-scaled GEMM)",
            "value": tf(ms) * world, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": {"workload": f"mm_mxfp8-{M}x{N}x{K}", "M": M, "N": N, "K": K,
                       "gemm": ("mxfp8_gemm_skinny_kernel: tcgen05 cta_group::2 "
                                "kind::mxf8f6f4 block-scaled (E4M3 x E4M3, UE8M0 per 32), "
                                "operands swapped (the weight's 256-row block is the MMA's M, "
                                "the activation rows its N), K split over the CTA pairs of a "
                                "cluster when output blocks are few"
                                if M <= 128 else
                                "mxfp8_gemm_kernel: tcgen05 cta_group::2 kind::mxf8f6f4 "
                                "block-scaled (E4M3 x E4M3, UE8M0 per 32), 256x256 tiles per "
                                "CTA pair, float32 accumulation in tensor memory, TMA-store "
                                "bf16 epilogue"),
                       "l2": ("operands fit in L2 (%.0f MB): a 256 MB memset and a 256 MB "
                              "read flush L2 before every timed launch, outside its events"
                              % (in_bytes / 1e6)
                              if flush is not None else
                              "operands larger than L2 (%.0f MB); no flush" % (in_bytes / 1e6))},
            "roofline": roof,
            "clocks": clk, "gpu_launches": 2 * args.steps, **extra}), flush=True)
    return 0


def main():
    args = parse()
    world, rank, local, pg = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.mm:
        return run_mm(args, world, rank, local, pg)

    import numpy as np
    import torch

    import mxfp8_block_scaled_rmsnorm_gb300 as mx
    from mxfp8_block_scaled_rmsnorm_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    mx.library()

    wl, R, C = load_workload(args)
    t = wl.tensors[0]
    step_bytes = wl.algorithmic_bytes()
    if args.residual and not wl.fused:
        raise SystemExit("--residual needs a fused workload")

    def host(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)

    x_host = [host(tt.x) for tt in wl.tensors]
    g_host = [host(tt.gamma) for tt in wl.tensors] if wl.fused else []
    xs = [h.to(device) for h in x_host]
    gs = [h.to(device) for h in g_host]
    outs = [mx.make_outputs(xx, wl.fused, wl.rowwise, wl.columnwise, args.scale_layout)
            for xx in xs]
    res_in, res_out = [], []
    if args.residual:
        rng = np.random.default_rng(100)
        for tt in wl.tensors:
            r = W.to_bf16_bits(rng.standard_normal(tt.x.shape, dtype=np.float32))
            res_in.append(host(r).to(device))
            res_out.append(torch.empty_like(res_in[-1]))
        # read the residual (2 B) and write h (2 B) per element
        step_bytes += sum(4 * tt.x.size for tt in wl.tensors)
    stream = torch.cuda.current_stream(device)
    eps = [tt.eps for tt in wl.tensors]
    offs = [tt.offset for tt in wl.tensors]

    if args.update:
        # the planes to install: the workload's own MXFP8 planes, compact
        srcs = [mx.quant_mxfp8(xx) for xx in xs]
        dsts = [mx.make_outputs(xx, False, True, True, "padded") for xx in xs]
        torch.cuda.synchronize(device)
        # read and write each code plane (1 B) and each scale plane (1/32 B)
        step_bytes = sum(2 * 2 * (tt.x.size + tt.x.size // 32) for tt in wl.tensors)

    def call(on_stream=None):
        if args.update:
            mx.update_planes(srcs, dsts, True, True, scale_layout="padded", stream=on_stream)
        elif args.residual:
            mx.add_rmsnorm_quant_mxfp8(xs, res_in, gs, eps, offs, wl.rowwise, wl.columnwise,
                                       out=outs, residual_out=res_out, stream=on_stream,
                                       scale_layout=args.scale_layout)
        elif wl.fused:
            mx.rmsnorm_quant_mxfp8(xs, gs, eps, offs, wl.rowwise, wl.columnwise, out=outs,
                                   stream=on_stream, scale_layout=args.scale_layout)
        else:
            mx.quant_mxfp8(xs, wl.rowwise, wl.columnwise, out=outs, stream=on_stream,
                           scale_layout=args.scale_layout)

    if args.graph:
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                call()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()          # the library launches on the capturing (current) stream
        torch.cuda.synchronize(device)
        step = graph.replay
    else:
        def step():
            call(stream)

    clocks = ClockSampler(device.index)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(device)
    # keep the GPU loaded long enough for the clock sampler to see it before
    # the timed region (untimed extra warm-up)
    clocks.mark("load")
    t_settle = time.time() + 0.4
    while time.time() < t_settle:
        for _ in range(20):
            step()
        torch.cuda.synchronize(device)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    flush = L2Flush(device) if fits_l2(wl) else None
    barrier(pg, device)
    torch.cuda.synchronize(device)
    clocks.mark("start")
    for i in range(args.steps):
        if flush is not None:
            flush(stream)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(device)
    clocks.mark("end")
    barrier(pg, device)
    clk = clocks.stop()

    per_launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    # with L2 flushes between launches the whole-job time is the launches' sum
    total_ms = sum(per_launch_ms) if flush is not None else starts[0].elapsed_time(ends[-1])
    total_ms = max_over_ranks(total_ms, pg, device)
    ms_per_step = total_ms / args.steps
    value = step_bytes * args.steps * world / (total_ms * 1e-3) / 1e9
    avg_launch_ms = sum(per_launch_ms) / len(per_launch_ms)
    achieved = step_bytes / (avg_launch_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak()

    # end to end: pinned host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        xh = [h.pin_memory() for h in x_host]
        gh = [h.pin_memory() for h in g_host]
        rh = [r.cpu().pin_memory() for r in res_in]
        pairs = [(v.cpu().pin_memory(), v) for o in outs for v in o if v is not None]
        pairs += [(r.cpu().pin_memory(), r) for r in res_out]
        h2d = sum(h.numel() * 2 for h in xh + gh + rh)
        d2h = sum(hv.numel() * hv.element_size() for hv, _ in pairs)

        def e2e_step():
            for d, h in zip(xs + gs + res_in, xh + gh + rh):
                d.copy_(h, non_blocking=True)
            step()
            for hv, dv in pairs:
                hv.copy_(dv, non_blocking=True)
            torch.cuda.synchronize(device)

        path = ("pinned host -> device copy, the C ABI call, device -> pinned host copy of "
                "every output, sync per step")
        pipelined = (wl.fused and len(wl.tensors) == 1 and not args.residual
                     and not args.update and not args.graph)
        if pipelined:
            # rows are independent in 32-row blocks, so the step can run in row
            # chunks: copy chunk i+1 in || compute chunk i || copy chunk i-1 out
            # (three streams; the results are byte-identical to one call)
            n_chunks = 16
            cr = -(-R // n_chunks // 32) * 32
            chunks = [(r0, min(R, r0 + cr)) for r0 in range(0, R, cr)]
            s_in, s_cmp, s_out = (torch.cuda.Stream(device) for _ in range(3))
            o = outs[0]
            present = [f for f in o._fields if getattr(o, f) is not None]
            host_of = dict(zip(present, (hv for hv, _ in pairs)))

            def rows_of(f, r0, r1):
                # s_col has one row per 32-row block
                return slice(r0 // 32, r1 // 32) if f == "s_col" else slice(r0, r1)

            def e2e_step():
                with torch.cuda.stream(s_in):
                    gs[0].copy_(gh[0], non_blocking=True)
                for r0, r1 in chunks:
                    with torch.cuda.stream(s_in):
                        xs[0][r0:r1].copy_(xh[0][r0:r1], non_blocking=True)
                    s_cmp.wait_stream(s_in)
                    view = mx.NormQuantOut(**{
                        f: (getattr(o, f)[rows_of(f, r0, r1)] if f in host_of else None)
                        for f in o._fields})
                    mx.rmsnorm_quant_mxfp8(xs[0][r0:r1], gs[0], t.eps, t.offset, wl.rowwise,
                                           wl.columnwise, out=[view], stream=s_cmp)
                    s_out.wait_stream(s_cmp)
                    with torch.cuda.stream(s_out):
                        for f, hv in host_of.items():
                            if f not in ("s_row", "s_col"):
                                hv[rows_of(f, r0, r1)].copy_(getattr(view, f), non_blocking=True)
                # the scale planes (1/32 of the codes) in one copy each at the
                # end: per-chunk copies of them cost more than their bytes
                with torch.cuda.stream(s_out):
                    for f in ("s_row", "s_col"):
                        if f in host_of:
                            host_of[f].copy_(getattr(o, f), non_blocking=True)
                torch.cuda.synchronize(device)

            path = ("pinned host -> device copies, rmsnorm_quant_mxfp8 (C ABI), device -> "
                    f"pinned host copies of every output, in {len(chunks)} row chunks on three "
                    "streams (copy in || compute || copy out; the scale planes copied once "
                    "after the last chunk), sync per step")

        for _ in range(2):
            e2e_step()
        n_e2e = max(3, min(args.steps, 20))
        barrier(pg, device)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        el = max_over_ranks(time.perf_counter() - t0, pg, device)
        e2e = {"value": step_bytes * n_e2e * world / el / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": n_e2e, "ms_per_step": el * 1e3 / n_e2e, "path": path}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and wl.fused and len(wl.tensors) == 1:
        rows = min(R, max(32, args.cpu_rows // 32 * 32))
        el = time_oracle(t, rows, wl.rowwise, wl.columnwise)
        sb = W.algorithmic_bytes(rows, C, True, wl.rowwise, wl.columnwise)
        # one thread on an eighth of the rows (the same per-row work)
        rows1 = min(rows, max(32, rows // 8 // 32 * 32))
        el1 = time_oracle(t, rows1, wl.rowwise, wl.columnwise, threads=1)
        sb1 = W.algorithmic_bytes(rows1, C, True, wl.rowwise, wl.columnwise)
        cpu = {"value": sb / el / 1e9, "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"rows 0-{rows - 1} of {R} ({100.0 * rows / R:.1f}% of the workload), "
                         f"all {C} columns, fused, one pass, {el:.2f} s wall",
               "single_thread": {"value": sb1 / el1 / 1e9, "unit": "GB/s", "cores": 1,
                                 "sample": f"rows 0-{rows1 - 1}, all {C} columns, fused, "
                                           f"one pass, {el1:.2f} s wall"},
               "cpu_model": cpu_model(), "arch": platform.machine()}

    if rank == 0:
        rec = base_record(args, wl, R, C, world)
        rec["config"]["algorithmic_bytes_per_step"] = step_bytes
        rec.update({
            "value": value,
            "ms_per_step": ms_per_step,
            "pct_of_peak": 100.0 * achieved / peak,
            # the same against GB300's nominal HBM3e figure (about 8 TB/s);
            # the roofline fraction uses the measured copy peak
            "pct_of_nominal_peak": 100.0 * achieved / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": (profiled_traffic(R, C) if args.workload in (0, 4)
                                     and args.scale_layout == "compact" and not args.residual
                                     and not args.update and wl.rowwise and wl.columnwise
                                     else None),
                         "kernel": ("update_planes_kernel" if args.update else
                                    "fused_rmsnorm_quant_kernel" if wl.fused else "quant_kernel"),
                         "variant": ("residual " if args.residual else "") + args.scale_layout,
                         "avg_launch_us": avg_launch_ms * 1e3,
                         # steady state; the first launch after the synchronize
                         # that opens the timed region runs from an idle GPU
                         "median_launch_us": statistics.median(per_launch_ms) * 1e3},
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": args.steps,
            "clocks": clk,
        })
        print(json.dumps(rec), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
