#!/usr/bin/env python3
"""Benchmark: SGEMM TFLOP/s at M=N=K=4096 (FP32, row-major, alpha=1.5, beta=0.5,
A, B, C uniform[-1,1) from seed 1) on GB300, as a fraction of the FP32 FFMA peak.

One step = one C = alpha*A*B + beta*C call of the library on operands already
resident in HBM. Prints ONE JSON line (rank 0). ``--impl reference`` times the
FP64 CPU oracle instead (a bounded sample of the same workload per step).

Multi-GPU: the path does not shard across GPUs here; ``--gpus N`` under
torchrun runs N independent replicas (weak scaling), max time over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import traceback
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SGEMM TFLOP/s at M=N=K=4096 FP32 and % of GB300 FP32 FFMA peak"
WORKLOAD = "square4096"
L2_BYTES = 126 * 2**20  # GB300 L2 (nvidia-smi reports ~126 MiB)
KERNEL_SOURCES = ["dense_fp32_gemm_04_gb300/csrc/ffma_kernels.cu", "dense_fp32_gemm_04_gb300/csrc/device_ptx.cuh",
                  "dense_fp32_gemm_04_gb300/csrc/schedule.cuh", "dense_fp32_gemm_04_gb300/csrc/tile_table.h"]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "ffma_sgemm_4096_traffic.md")
TRAFFIC_WORKLOAD = "square4096"  # the workload that capture was taken on


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    from dense_fp32_gemm_04_gb300 import inputs

    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(inputs.PROBLEMS),
                    help="configured problem timed as the headline (default: %(default)s)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--tf32-steps", type=int, default=50, help="calls timed in the flagged TF32 mode (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other configured problem sizes")
    ap.add_argument("--no-context", action="store_true", help="skip the cuBLAS context timing")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed
class World:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.size = int(os.environ.get("WORLD_SIZE", "1"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False

    def init(self, backend):
        if self.size > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist

            dist.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        import torch.distributed as dist

        dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist

            dist.destroy_process_group()


def aggregate(per_rank_seconds, flops_per_rank):
    """Whole-job throughput: all ranks' flops over the slowest rank's time (TFLOP/s)."""
    t = max(per_rank_seconds)
    return sum(flops_per_rank) / t / 1e12, t


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if t0 is not None and (ts < t0 or ts > t1 + 0.2):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def gemm_flops(M, N, K):
    """FLOPs of one C = alpha*A*B + beta*C: K multiplies and K adds per output (2MNK)."""
    return 2.0 * M * N * K


def operand_load_bytes(M, N, K, BM, BN):
    """Bytes a BM x BN tiling loads from L2/HBM for A and B: K * (1/BM + 1/BN) floats per output."""
    return 4.0 * M * N * K * (1.0 / BM + 1.0 / BN)


def smem_reads_per_output(K, TM, TN=1):
    """Shared-memory reads per output of a TM x TN register microtile: K * (TM + TN) / (TM * TN)."""
    return K * (TM + TN) / (TM * TN)


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and with runs of whitespace collapsed (string
    and character literals kept), so that a comment edit does not change the hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the FP32 kernel's code (comments excluded) that a traffic capture was taken on."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel source."""
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None
    m_hash = re.search(r"^kernel_source_sha256_16:\s*([0-9a-f]+)", text, re.M)
    m_val = re.search(r"^dram_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_val.group(1))


def problem(name):
    from dense_fp32_gemm_04_gb300 import inputs

    p = dict(inputs.PROBLEMS[name])
    return p


def cpu_oracle_sample(name, seconds, A=None, B=None, C=None, nthreads=0):
    """Time the FP64 oracle on rows of the workload for about ``seconds`` (``nthreads`` 0: all host threads)."""
    import numpy as np

    import oracle
    from dense_fp32_gemm_04_gb300 import inputs

    p = problem(name)
    if A is None:
        A, B, C = inputs.problem_operands(name)
    M, N, K = p["M"], p["N"], p["K"]
    threads = nthreads or oracle.max_threads()
    rows_done, elapsed, r, lo = 0, 0.0, 1, 0
    while elapsed < seconds:
        rows = np.arange(lo, min(M, lo + r))
        t = time.perf_counter()
        oracle.sgemm_f64(A, B, C, p["alpha"], p["beta"], rows=rows, with_mag=False, nthreads=nthreads)
        dt = time.perf_counter() - t
        elapsed += dt
        rows_done += len(rows)
        lo = (lo + len(rows)) % M  # small problems are repeated until the budget is spent
        # grow the batch toward the remaining budget
        per_row = dt / len(rows)
        r = max(1, min(M, int((seconds - elapsed) / max(per_row, 1e-9)) + 1, 4 * r))
    flops = 2.0 * rows_done * N * K
    return {"value": flops / elapsed / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows_done} rows (C has {M}) for {shape_text(M, N, K)} ({rows_done}x{N}x{K} MACs, FP64 "
                      f"accumulate, i-k-j loop, {threads} threads), {elapsed:.1f} s"}


def cpu_oracle_configs(seconds_each, C2=None):
    """The oracle's GFLOP/s at 1 thread and at all host threads on the 256^3, 4096^3, ragged and skinny problems."""
    import oracle

    out = []
    for name in ("square256", "square4096", "ragged", "skinny_tall"):
        ops = C2 if (name == "square4096" and C2 is not None) else (None, None, None)
        for nt in (1, oracle.max_threads()):
            d = cpu_oracle_sample(name, seconds_each, *ops, nthreads=nt)
            out.append({"problem": name, "threads": nt, "gflops": d["value"] * 1e3, "sample": d["sample"]})
    return out


def workload_text(p):
    dist = {"uniform": "uniform[-1,1)", "normal": "N(0,1)", "int": "int{-2..2}", "zero": "0"}
    da, db, dc = (dist[d] for d in p["dist"])
    ops = f"A,B,C {da}" if da == db == dc else f"A {da}, B {db}, C {dc}"
    return (f"sgemm {shape_text(p['M'], p['N'], p['K'])} alpha={p['alpha']} beta={p['beta']} {ops} "
            f"seed {p['seed']}")


def shape_text(M, N, K):
    return f"M=N=K={K}" if M == N == K else f"M={M} N={N} K={K}"


# ---------------------------------------------------------------- reference arm
def run_reference(args, world):
    if world.rank != 0:
        return 0
    import numpy as np

    import oracle
    from dense_fp32_gemm_04_gb300 import inputs

    p = problem(args.workload)
    A, B, C = inputs.problem_operands(args.workload)
    M, N, K = p["M"], p["N"], p["K"]
    rows_per_step = 8
    threads = oracle.max_threads()

    def step(i):
        lo = (i * rows_per_step) % M
        rows = np.arange(lo, min(M, lo + rows_per_step))
        oracle.sgemm_f64(A, B, C, p["alpha"], p["beta"], rows=rows, with_mag=False)
        return len(rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    rows = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_text(p),
                   "step": f"{rows_per_step} rows of C per step (bounded sample of the workload)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_per_step} of {M} rows of C per step, FP64 i-k-j oracle, {threads} threads"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def measured_bf16_peak():
    """Dense bf16 TFLOP/s measured on this GPU model (burst), or the stated fallback."""
    try:
        d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def measure_min2(torch, sg, h, dA, dB, dC, M, N, K, alpha, beta, stream, ms_per_call, steps=20):
    """Cost of also returning C's two smallest elements (sgemm_run_min2) over a plain call."""
    C = dC.clone()
    for _ in range(3):
        h.run_min2(dA, dB, C, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        h.run_min2(dA, dB, C, alpha, beta, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    extra = max(ms - ms_per_call, 1e-6)
    return {"ms_per_call": ms, "extra_ms_over_sgemm_run": ms - ms_per_call,
            "reduction_gbs": 4.0 * M * N / (extra * 1e-3) / 1e9,
            "note": "two smallest elements of C with positions; the extra pass reads C once (HBM-bound)"}


def measure_tf32(torch, sg, dA, dB, dC, M, N, K, alpha, beta, stream, device, steps=50):
    """Time the flagged TF32 tensor-core mode on the same operands (outside the FP32 timed region)."""
    h = sg.Sgemm(device)
    h.set_math_mode(sg.MATH_TF32)
    C = dC.clone()
    for _ in range(3):
        h.run(dA, dB, C, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    st, code = h.check_device_status()
    plan = h.last_plan()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        h.run(dA, dB, C, alpha, beta, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    h.close()
    ms = e0.elapsed_time(e1) / steps
    achieved = gemm_flops(M, N, K) / (ms * 1e-3) / 1e12
    bf16, basis = measured_bf16_peak()
    peak = bf16 * (1.1 / 2.25)  # nominal dense tf32 : bf16 ratio
    kernel = ("tf32_kernel<true> (CTA pairs, tcgen05 .cta_group::2, 256 x 256 tiles)" if plan.config == 1
              else "tf32_kernel<false> (one CTA per 128 x 256 tile)")
    return {"value": achieved, "unit": "TFLOP/s", "ms_per_call": ms, "steps": steps, "status": st,
            "launches_per_call": plan.launches, "kernel": kernel,
            "plan": {k: plan.as_dict()[k] for k in ("config", "bm", "bn", "stages", "grid", "units", "sk_tiles",
                                                    "sk_grid")},
            "note": "flagged SGEMM_MATH_TF32 (TF32 inputs, FP32 accumulate); per-call time includes the stream-K reduction",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_basis": f"{basis} bf16 {bf16} TFLOP/s x 1.1/2.25 (nominal tf32:bf16 dense ratio)"}}


CONFIG_PROBLEMS = ["square256", "sweep512", "sweep1024", "sweep2048", "sweep8192", "sweep16384", "ragged",
                   "skinny_tall", "skinny_wide"]


def measure_configs(torch, sg, h, dev, stream, hbm_gbs, min_seconds=1.0):
    """TFLOP/s, % of the FFMA peak and algorithmic HBM GB/s of every other configured problem.

    Seeded operands of each problem; 5 warm-up calls, then at least 20 timed calls and at
    least ``min_seconds`` of them; L2 is flushed (a 256 MiB write) before every timed call
    and only the call itself sits between its CUDA events (median and min reported).
    Outside the headline timed region.
    """
    from dense_fp32_gemm_04_gb300 import inputs

    flush = torch.empty(64 * 2**20, dtype=torch.float32, device=dev)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "")) or None
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or "0"))
    rows = []
    sampler.start()
    t0 = time.time()
    for name in CONFIG_PROBLEMS:
        q = inputs.PROBLEMS[name]
        M, N, K, alpha, beta = q["M"], q["N"], q["K"], q["alpha"], q["beta"]
        A, B, C = inputs.problem_operands(name)
        dA, dB, dC = (torch.from_numpy(x).to(dev) for x in (A, B, C))
        del A, B, C
        flops = gemm_flops(M, N, K)
        for _ in range(5):
            h.run(dA, dB, dC, alpha, beta, stream=stream)
        times = []
        while len(times) < 20 or sum(times) < min_seconds * 1e3:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            for e0, e1 in ev:
                flush.fill_(1.0)
                e0.record(stream)
                h.run(dA, dB, dC, alpha, beta, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            times += [e0.elapsed_time(e1) for e0, e1 in ev]
        st, _ = h.check_device_status()
        plan = h.last_plan()
        ms = statistics.median(times)
        bytes_alg = 4.0 * (M * K + K * N + M * N * (2 if beta != 0 else 1))
        rows.append({"problem": name, "M": M, "N": N, "K": K, "alpha": alpha, "beta": beta, "calls": len(times),
                     "ms_median": ms, "ms_min": min(times), "tflops": flops / (ms * 1e-3) / 1e12,
                     "tflops_best": flops / (min(times) * 1e-3) / 1e12, "hbm_gbs": bytes_alg / (ms * 1e-3) / 1e9,
                     "flop_per_byte": flops / bytes_alg, "status": st,
                     "plan": {"config": plan.config, "splits": plan.splits, "sk_tiles": plan.sk_tiles,
                              "transpose_a": plan.transpose_a, "launches": plan.launches}})
        del dA, dB, dC
    t1 = time.time()
    sampler.stop()
    clocks = sampler.summary(t0, t1)
    sm_mhz = clocks["sm_mhz"] if clocks else None
    peak = nsm * 256 * sm_mhz * 1e-6 if sm_mhz else None
    ridge = (peak * 1e3 / hbm_gbs) if (peak and hbm_gbs) else None
    peak_max = nsm * 256 * clocks["sm_max_mhz"] * 1e-6 if clocks else None
    for r in rows:
        r["pct_ffma_peak"] = 100.0 * r["tflops"] / peak if peak else None
        r["pct_ffma_peak_at_max_clock"] = 100.0 * r["tflops"] / peak_max if peak_max else None
        r["pct_hbm"] = 100.0 * r["hbm_gbs"] / hbm_gbs if hbm_gbs else None
        r["bound"] = ("alu" if r["flop_per_byte"] >= ridge else "hbm") if ridge else None
    del flush
    torch.cuda.empty_cache()
    return {"problems": rows, "clocks": clocks, "ffma_peak_tflops": peak, "ffma_peak_tflops_at_max_clock": peak_max,
            "hbm_peak_gbs": hbm_gbs,
            "ridge_flop_per_byte": ridge,
            "note": "per-call CUDA events, L2 flushed before each call, rates from the median call; peak at the "
                    "median SM clock sampled here; hbm_gbs = algorithmic bytes (A, B, C written, C read when "
                    "beta != 0) / time"}


def measure_library_context(torch, dA, dB, dC, alpha, beta, flops, steps=20):
    """cuBLAS through torch.addmm on the same operands (C <- alpha*A*B + beta*C), FP32 and
    TF32: context only, never on the product path."""
    out = {"note": "torch.addmm (cuBLAS) on the same operands, alpha/beta included; context only"}
    prev = torch.backends.cuda.matmul.allow_tf32
    D = torch.empty_like(dC)
    try:
        for mode, tf32 in (("fp32", False), ("tf32", True)):
            torch.backends.cuda.matmul.allow_tf32 = tf32
            for _ in range(3):
                torch.addmm(dC, dA, dB, beta=beta, alpha=alpha, out=D)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                torch.addmm(dC, dA, dB, beta=beta, alpha=alpha, out=D)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / steps
            out[f"{mode}_tflops"] = flops / (ms * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    del D
    return out


def measured_hbm_gbs():
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


# ---------------------------------------------------------------- our arm
def optional(name, fn, *a, **kw):
    """Run an optional section of the line (min2, configs, context, TF32, CPU baseline):
    a failure there becomes {"error": ...} in its key (traceback on stderr) instead of
    costing the headline measurement."""
    try:
        return fn(*a, **kw)
    except Exception as e:  # noqa: BLE001 - reported in the JSON line and on stderr
        traceback.print_exc(file=sys.stderr)
        return {"error": f"{name}: {type(e).__name__}: {e}"}


def run_ours(args, world):
    import numpy as np
    import torch

    import dense_fp32_gemm_04_gb300 as sg
    from dense_fp32_gemm_04_gb300 import _build, inputs

    _build.build()
    torch.cuda.set_device(world.local_rank)
    dev = torch.device("cuda", world.local_rank)
    world.init("nccl" if world.size > 1 else "gloo")

    p = problem(args.workload)
    M, N, K, alpha, beta = p["M"], p["N"], p["K"], p["alpha"], p["beta"]
    A, B, C = inputs.problem_operands(args.workload)
    dA, dB, dC = (torch.from_numpy(x).to(dev) for x in (A, B, C))
    h = sg.Sgemm(world.local_rank)
    stream = torch.cuda.current_stream(dev)
    flops = gemm_flops(M, N, K)
    operand_bytes = 4 * (M * K + K * N + M * N)

    for _ in range(max(3, args.warmup)):
        h.run(dA, dB, dC, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    st, code = h.check_device_status()
    if st != sg.SGEMM_OK:
        raise RuntimeError(f"device status {code:#x} after warm-up")
    plan = h.last_plan()

    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "")) or None
    sampler = ClockSampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(world.local_rank)))
    sampler.start()

    # Operands that fit in L2 would be timed warm: flush it (a 256 MiB write) before every
    # call and take the time from the per-call events alone.
    flush = torch.empty(64 * 2**20, dtype=torch.float32, device=dev) if operand_bytes <= L2_BYTES else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    world.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(1.0)
        starts[i].record(stream)
        h.run(dA, dB, dC, alpha, beta, stream=stream)
        ends[i].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    world.barrier()
    t_wall1 = time.time()
    sampler.stop()
    elapsed = ev0.elapsed_time(ev1) / 1e3
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if flush is not None:
        elapsed = sum(kernel_ms) / 1e3  # the flushes between calls are not GEMM time
        del flush
    st, code = h.check_device_status()
    if st != sg.SGEMM_OK:
        raise RuntimeError(f"device status {code:#x} in the timed region")

    t_max = world.max(elapsed)
    value = flops * args.steps * world.size / t_max / 1e12

    # End to end through the host-buffer entry point: pinned host operands,
    # H2D of A, B, C and D2H of C inside every step.
    pA, pB = (torch.from_numpy(x).pin_memory() for x in (A, B))
    pC = torch.from_numpy(C).pin_memory()
    h.run_host(pA, pB, pC, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    e2e_steps = max(3, args.e2e_steps)
    world.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        h.run_host(pA, pB, pC, alpha, beta, stream=stream)
    torch.cuda.synchronize()
    e2e_t = world.max(time.perf_counter() - t0)
    e2e_value = flops * e2e_steps * world.size / e2e_t / 1e12

    min2 = optional("min2", measure_min2, torch, sg, h, dA, dB, dC, M, N, K, alpha, beta, stream,
                    ms_per_call=elapsed / args.steps * 1e3)
    configs = (optional("configs", measure_configs, torch, sg, h, dev, stream, measured_hbm_gbs())
               if world.size == 1 and not args.no_configs else None)
    library = (optional("library_context", measure_library_context, torch, dA, dB, dC, alpha, beta, flops)
               if world.size == 1 and not args.no_context else None)
    tf32 = (optional("tf32_mode", measure_tf32, torch, sg, dA, dB, dC, M, N, K, alpha, beta, stream,
                     world.local_rank, args.tf32_steps)
            if args.tf32_steps > 0 else None)

    clocks = sampler.summary(t_wall0, t_wall1)
    nsm = props.multi_processor_count
    avg_kernel_s = statistics.fmean(kernel_ms) / 1e3
    achieved = flops / avg_kernel_s / 1e12
    sm_mhz = clocks["sm_mhz"] if clocks else None
    peak = nsm * 128 * 2 * sm_mhz * 1e6 / 1e12 if sm_mhz else None
    roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if peak else None,
                "traffic": recorded_traffic() if args.workload == TRAFFIC_WORKLOAD else None,
                "kernel": ("ffma_sgemm_kernel (plan config %d, %dx%d tile, A %s)" %
                           (plan.config, plan.bm, plan.bn, "transposed first" if plan.transpose_a else "as given")) +
                          (" + transpose_kernel (A^T)" if plan.transpose_a else "") +
                          (" + sk_reduce_kernel" if plan.sk_tiles > 0 else "") +
                          (" + splitk_reduce_kernel" if plan.splits > 1 else "") +
                          (" (timed together per call: a lower bound for the mainloop)" if plan.launches > 1 else ""),
                "peak_basis": f"{nsm} SMs x 128 FP32 FMA/clk x 2 FLOP x median SM clock under load "
                              f"({sm_mhz} MHz, nvidia-smi during the timed region)",
                "frac_at_max_clock": (achieved / (nsm * 256 * clocks["sm_max_mhz"] * 1e-6)) if clocks else None}

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world.size, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_text(p),
                   "M": M, "N": N, "K": K, "layout": "row-major",
                   "l2": (f"no flush: operands {operand_bytes / 2**20:.0f} MiB > L2 {L2_BYTES / 2**20:.0f} MiB"
                          if operand_bytes > L2_BYTES else
                          f"operands {operand_bytes / 2**20:.0f} MiB fit in L2: 256 MiB flush before every call, "
                          "time from the per-call events"),
                   "parallelism": f"replicas x{world.size}", "plan": plan.as_dict(),
                   "operand_load_bytes_model": operand_load_bytes(M, N, K, plan.bm, plan.bn)},
        "pct_fp32_ffma_peak": (100.0 * achieved / peak) if peak else None,
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 4 * (M * K + K * N + M * N),
                "d2h_bytes_per_step": 4 * M * N, "steps": e2e_steps, "api": "sgemm_run_host (pinned host buffers)"},
        "gpu_launches": plan.launches * args.steps,
        "clocks": clocks,
        "tf32_mode": tf32,
        "min2": min2,
        "configs": configs,
        "library_context": library,
    }
    if world.rank == 0 and world.size == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = optional("cpu_baseline", cpu_oracle_sample, args.workload, args.cpu_seconds, A, B, C)
        if not args.no_configs and "error" not in line["cpu_baseline"]:
            line["cpu_baseline"]["configs"] = optional(
                "cpu_baseline.configs", cpu_oracle_configs, min(2.0, args.cpu_seconds / 4),
                (A, B, C) if args.workload == "square4096" else None)
    if world.rank == 0:
        print(json.dumps(line), flush=True)
    h.close()
    world.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    world = World()
    if args.impl == "reference":
        return run_reference(args, world)
    return run_ours(args, world)


if __name__ == "__main__":
    sys.exit(main())
