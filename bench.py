#!/usr/bin/env python3
"""Benchmark: single-precision dense GEMM C = A @ B (row-major) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--algo auto|ffma|3xtf32]
                    [--workload square_8192_normal] [--impl ours|reference]

One step is one call of the library's public entry point (operand staging,
the GEMM kernel and any split-K reduction, all on the GPU) on the 8192^3
workload with N(0,1) inputs.  The inputs (2 x 256 MiB) are larger than the
129 MB L2, so no flush is needed between steps; smaller workloads get an L2
flush (a 512 MiB write) between timed steps, outside the timed pairs.

Timing follows the lecture-12 benchmark helper and the cuda-gemm README's
method: CUDA events per step on the launching stream after warm-up, device
memory allocated once.  Printed as ONE JSON line by rank 0.

--impl reference times the CPU oracle (the double-accumulation triple loop)
on the host cores instead, each step a bounded sample of rows of the same
workload.  Under torchrun (N > 1) every rank runs an independent replica
(the operation has no data exchange), the time is the max over ranks and
the value is the total work of all ranks over that time.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP32 GEMM TFLOPS at M=N=K=8192 on 1 GB300 and % of FP32/tensor roofline"
UNIT = "TFLOPS"
L2_BYTES = 129 * 1000 * 1000
# nominal dense tensor rates of the part (context for scaling a measured peak)
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_TF32_TFLOPS = 1100.0
SUSTAINED_S = 2.0  # timed regions longer than this are scored against the sustained peak
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
FFMA_LANES_PER_SM = 128  # FP32 FMA units per SM (4 sub-partitions x 32)
# The tensor core's own tf32 ceiling on this part, measured by a
# microbenchmark (one lane per SM pair issuing back-to-back cta_group::2
# kind::tf32 M256 N256 K8 MMAs on shared-memory-resident tiles, no TMA, no
# epilogue, 3.15 ms): 1215 TFLOP/s tf32, i.e. 405 of 3xTF32-effective work.
# Reported beside the prescribed roofline, whose denominator scales the
# measured bf16 rate by the nominal tf32/bf16 ratio and so reads above 1.
TF32_CEILING_TFLOPS = 1215.0


# ---------------------------------------------------------------------------
# distributed plumbing (harness only: nothing of the GEMM is exchanged)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist

    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a scalar over all ranks (identity for a single process)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# peaks and clocks
# ---------------------------------------------------------------------------
def load_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock, power and throttle reasons in the background."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None
        self.c0 = None

    COUNTERS = ["clocks_event_reasons_counters.sw_power_cap",
                "clocks_event_reasons_counters.sw_thermal_slowdown",
                "clocks_event_reasons_counters.hw_thermal_slowdown"]

    def counters(self) -> list | None:
        """Microseconds each clock-reducing reason has been active (None if unknown).

        nvidia-smi's sampled readings lag a timed region of a few hundred
        milliseconds; these running totals, read before and after it, do not.
        """
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.COUNTERS), "--format=csv,noheader,nounits"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            out = subprocess.run(cmd, capture_output=True, text=True, timeout=10).stdout
            return [float(x) for x in out.strip().splitlines()[0].split(",")]
        except (OSError, ValueError, IndexError, subprocess.SubprocessError):
            return None

    def start(self):
        self.c0 = self.counters()
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,nounits",
                   "-lms", "100"]
            if self.gpu_id:
                cmd += ["-i", self.gpu_id]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        summary = self.summarise(text)
        c1 = self.counters()
        if self.c0 is not None and c1 is not None:
            names = ["sw_power_cap", "sw_thermal_slowdown", "hw_thermal_slowdown"]
            active_us = {n: max(0.0, b - a) for n, a, b in zip(names, self.c0, c1)}
            summary["reason_active_us"] = active_us
            summary["reasons"] = sorted(set(summary["reasons"]) |
                                        {n for n, v in active_us.items() if v > 0})
        return summary

    @staticmethod
    def summarise(text: str) -> dict:
        rows = [r for r in csv.reader(io.StringIO(text)) if r and not r[0].startswith("index")]
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": sorted(reasons), "samples": 0}
        loaded = [s for s, p in zip(sm, pw) if p >= 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw)}


KERNEL_SOURCES = {
    "sgemm_ffma": ["sgemm_ffma.cu", "device_sync.cuh"],
    "sgemm_3xtf32": ["sgemm_3xtf32.cu", "tf32x3_common.cuh", "device_sync.cuh", "tcgen05.cuh"],
    "sgemm_3xtf32_tmem": ["sgemm_3xtf32_tmem.cu", "tf32x3_common.cuh", "device_sync.cuh",
                          "tcgen05.cuh"],
    "sgemm_3xtf32_tmem_pair": ["sgemm_3xtf32_tmem.cu", "tf32x3_common.cuh", "device_sync.cuh",
                               "tcgen05.cuh"],
    "sgemm_3xtf32_tmem_wide": ["sgemm_3xtf32_tmem.cu", "tf32x3_common.cuh", "device_sync.cuh",
                               "tcgen05.cuh"],
}


def source_digest(kernel: str) -> str:
    """Digest of a kernel's device sources: ties stored ncu counters to the code they measured."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_gemm_row_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    e = table.get(kernel, {}).get(workload)
    if not e or e.get("source_digest") != source_digest(kernel):
        return None
    return float(e["dram_bytes_per_launch"])


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline arm)
# ---------------------------------------------------------------------------
def oracle_rows_timing(A, B, seconds: float, single_thread: bool = False) -> dict:
    """Time the oracle on the first R rows of C, R sized to take ~`seconds`.

    A warm-up pass on a few rows (page-in, thread start) is followed by a
    calibration pass; R is a multiple of the oracle's thread count so that
    every thread gets the same number of rows.  single_thread: the oracle on
    one host thread.
    """
    import oracle

    M, K = A.shape
    N = B.shape[1]
    nt = 1 if single_thread else 0  # 0: all of the oracle's threads
    threads = 1 if single_thread else max(1, oracle.max_threads())
    oracle.ref_gemm_rows(A, B, 0, min(M, threads), nthreads=nt)  # warm-up
    cal = min(M, 2 * threads)
    t0 = time.perf_counter()
    oracle.ref_gemm_rows(A, B, 0, cal, nthreads=nt)
    per_row = max(time.perf_counter() - t0, 1e-6) / cal
    rows = int(seconds / per_row) // threads * threads
    rows = int(max(threads, min(M, rows)))
    rows = min(rows, M)
    t0 = time.perf_counter()
    oracle.ref_gemm_rows(A, B, 0, rows, nthreads=nt)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"rows": rows, "seconds": dt, "flops": flops, "tflops": flops / dt / 1e12,
            "cores": threads}


def cublas_context(a, b, steps: int = 10) -> float | None:
    """cuBLAS SGEMM (torch.matmul, TF32 off) on the same device tensors: context only."""
    import torch

    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = False
        for _ in range(3):
            c = a @ b
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            c = a @ b
        e1.record()
        torch.cuda.synchronize()
        del c
        ms = e0.elapsed_time(e1) / steps
        return 2.0 * a.shape[0] * a.shape[1] * b.shape[1] / (ms * 1e-3) / 1e12
    except Exception:
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def run_reference(args, world, rank):
    """--impl reference: the CPU oracle as it stands, bounded rows per step."""
    import oracle
    from seeded_inputs import workload_by_name, make_workload

    if rank != 0:
        return 0
    w = workload_by_name(args.workload)
    A, B = make_workload(w)
    budget = min(10.0, 150.0 / max(1, args.steps + args.warmup))
    cal = oracle_rows_timing(A, B, budget)
    rows = cal["rows"]
    for _ in range(args.warmup):
        oracle.ref_gemm_rows(A, B, 0, rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ref_gemm_rows(A, B, 0, rows)
        times.append(time.perf_counter() - t0)
    flops = 2.0 * rows * w.N * w.K
    total = sum(times)
    value = flops * len(times) / total / 1e12
    sample = (f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} product ({rows * w.N} of "
              f"{w.M * w.N} outputs, full K) per step")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cal["cores"], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import dense_fp32_gemm_row_gb300 as g
    from seeded_inputs import make_workload, workload_by_name

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    g.load()

    w = workload_by_name(args.workload)
    algo = g.ALGOS[args.algo]
    M, N, K = w.M, w.N, w.K
    A_np, B_np = make_workload(w)
    a = torch.from_numpy(A_np).to(dev)
    b = torch.from_numpy(B_np).to(dev)
    c = torch.empty((M, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    st, plan = g.gemm_f32_plan(M, N, K, algo, args.splits, a.data_ptr(), b.data_ptr(),
                               c.data_ptr())
    g.check(st, "plan")
    input_bytes = 4 * (M * K + K * N)
    flush = None
    if input_bytes <= L2_BYTES * 2:
        flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def step(ev_b=None, ev_e=None):
        st = g.gemm_f32_algo_splitk_ev(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K, algo,
                                       args.splits, stream.cuda_stream,
                                       ev_b.cuda_event if ev_b is not None else None,
                                       ev_e.cuda_event if ev_e is not None else None)
        g.check(st, "gemm_f32_algo_splitk_ev")

    K_steps = args.steps
    sb = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    se = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(K_steps)]
    for ev in sb + se + kb + ke:  # create the events so that their handles exist
        ev.record(stream)
    for _ in range(args.warmup):
        step()
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize(dev)
    g.check(g.gemm_f32_device_status(1), "device status after warm-up")

    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_uuid)
    sampler.start()
    time.sleep(0.3)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(K_steps):
        sb[i].record(stream)
        step(kb[i], ke[i])
        se[i].record(stream)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    g.check(g.gemm_f32_device_status(1), "device status after timed steps")

    step_ms = [sb[i].elapsed_time(se[i]) for i in range(K_steps)]
    kern_ms = [kb[i].elapsed_time(ke[i]) for i in range(K_steps)]

    # context for inputs that fit in L2: the same calls back to back without
    # the flush (the pages' convention: repeats on a warm cache); not the
    # reported value
    warm = None
    if flush is not None:
        for i in range(K_steps):
            sb[i].record(stream)
            step()
            se[i].record(stream)
        torch.cuda.synchronize(dev)
        warm_ms = statistics.median(sb[i].elapsed_time(se[i]) for i in range(K_steps))
        warm = {"step_ms_median": warm_ms,
                "tflops": 2.0 * M * N * K / (warm_ms * 1e-3) / 1e12,
                "note": "context: the same calls without the L2 flush between them"}
    if flush is None:
        total_ms = sb[0].elapsed_time(se[-1])
    else:
        total_ms = sum(step_ms)
    total_ms = reduce_max(total_ms, world, dev)
    flops = 2.0 * M * N * K
    value = flops * K_steps * world / (total_ms * 1e-3) / 1e12

    # roofline of the dominant kernel (the GEMM kernel itself)
    peaks, peak_src = load_peaks()
    kern_mean_s = statistics.mean(kern_ms) * 1e-3
    achieved = flops / kern_mean_s / 1e12
    props = torch.cuda.get_device_properties(dev)
    # a timed region of more than SUSTAINED_S seconds runs under the power
    # cap (measured: 1.37 kW, SM clock 1.86 GHz over 7.6 s of 8192^3 calls),
    # so its tensor peak is the sustained bf16 figure, else the burst one
    sustained = total_ms * 1e-3 > SUSTAINED_S
    peak_kind = "sustained" if sustained else "burst"
    if plan["algo"] == g.ALGO_3XTF32:
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        bf16 = float(peaks.get(key, FALLBACK_PEAKS[key]))
        peak = bf16 * (NOMINAL_TF32_TFLOPS / NOMINAL_BF16_TFLOPS) / 3.0
        bound = "tensor"
        form = {(256, 256): "_pair", (256, 128): "_wide"}.get(
            (plan["tile_m"], plan["tile_n"]), "")
        kname = "sgemm_3xtf32_tmem" + form if plan.get("b_in_tmem") else "sgemm_3xtf32"
    else:
        mhz = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2070.0)
        peak = props.multi_processor_count * FFMA_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        bound, kname = "alu", "sgemm_ffma"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": stored_traffic(kname, w.name),
                "kernel": kname, "peak_source": peak_src, "peak_kind": peak_kind}
    if bound == "tensor":
        ceiling = TF32_CEILING_TFLOPS / 3.0
        roofline["ceiling"] = {
            "value": ceiling, "frac": achieved / ceiling, "unit": "TFLOP/s",
            "source": "microbenchmark of back-to-back cta_group::2 kind::tf32 MMAs on this "
                      "part (1215 TFLOP/s tf32), / 3 products"}

    # the CUDA-core kernel on the same inputs, timed the same way right after
    # the timed region (its own short loop, outside it): the FFMA roofline
    ffma = None
    if plan["algo"] != g.ALGO_FFMA and not args.no_ffma:
        fb = [torch.cuda.Event(enable_timing=True) for _ in range(args.ffma_steps)]
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(args.ffma_steps)]

        def ffma_step(ev_b=None, ev_e=None):
            g.check(g.gemm_f32_algo_splitk_ev(a.data_ptr(), b.data_ptr(), c.data_ptr(), M, N, K,
                                              g.ALGO_FFMA, 0, stream.cuda_stream,
                                              ev_b.cuda_event if ev_b is not None else None,
                                              ev_e.cuda_event if ev_e is not None else None),
                    "ffma step")

        for _ in range(3):
            ffma_step()
        for ev in fb + fe:
            ev.record(stream)
        torch.cuda.synchronize(dev)
        for i in range(args.ffma_steps):
            ffma_step(fb[i], fe[i])
            if flush is not None:
                flush.zero_()
        torch.cuda.synchronize(dev)
        g.check(g.gemm_f32_device_status(1), "device status after the FFMA steps")
        fms = [fb[i].elapsed_time(fe[i]) for i in range(args.ffma_steps)]
        mhz = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or 2070.0)
        fpeak = props.multi_processor_count * FFMA_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        ftf = flops / (statistics.mean(fms) * 1e-3) / 1e12
        ffma = {"kernel": "sgemm_ffma", "kernel_ms_mean": statistics.mean(fms),
                "kernel_ms_median": statistics.median(fms), "steps": args.ffma_steps,
                "tflops": ftf, "peak": fpeak, "frac": ftf / fpeak, "bound": "alu",
                "note": "CUDA-core kernel on the same inputs, timed after the timed region"}

    # end to end through the public host-buffer entry point (pinned host
    # memory): every step copies A and B in and C out inside the call
    e2e_steps = max(1, min(args.e2e_steps, K_steps))
    hA = torch.from_numpy(A_np).pin_memory()
    hB = torch.from_numpy(B_np).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()

    def e2e_step():
        g.check(g.gemm_f32_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), M, N, K, algo,
                                stream.cuda_stream), "gemm_f32_host")

    for _ in range(2):
        e2e_step()
    eb = torch.cuda.Event(enable_timing=True)
    ee = torch.cuda.Event(enable_timing=True)
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    eb.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(eb.elapsed_time(ee), world, dev)
    e2e_value = flops * e2e_steps * world / (e2e_ms * 1e-3) / 1e12
    if not np.isfinite(hC[0, :8].numpy()).all():
        raise SystemExit("non-finite output")

    context = None
    if not args.no_context:
        context = {"cublas_sgemm_tflops": cublas_context(a, b),
                   "note": "torch.matmul fp32 with TF32 disabled, same inputs, not linked"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_rows_timing(A_np, B_np, args.cpu_seconds)
        cpu = {"value": cb["tflops"], "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
               "sample": (f"rows 0..{cb['rows'] - 1} of the {M}x{N}x{K} product "
                          f"({cb['rows'] * N} outputs, full K, {cb['seconds']:.1f} s)")}
        if 2.0 * M * N * K <= 2.0 * 2048 ** 3:
            # the small workloads also on one host thread
            c1 = oracle_rows_timing(A_np, B_np, min(args.cpu_seconds, 10.0), single_thread=True)
            cpu["single_thread"] = {
                "value": c1["tflops"], "unit": UNIT, "cores": 1,
                "sample": (f"rows 0..{c1['rows'] - 1} of the product "
                           f"({c1['rows'] * N} outputs, full K, {c1['seconds']:.1f} s)")}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K_steps,
        "warmup": args.warmup, "ms_per_step": total_ms / K_steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "M": M, "N": N, "K": K, "dist": w.dist,
                   "algo": {1: "ffma", 2: "3xtf32"}.get(plan["algo"], str(plan["algo"])),
                   "splits": plan["splits"], "tile": [plan["tile_m"], plan["tile_n"],
                                                      plan["tile_k"]],
                   "stages": plan["stages"], "ctas": plan["ctas"],
                   "l2": ("flush 512 MiB between steps" if flush is not None
                          else "inputs larger than L2, no flush"),
                   "parallelism": f"replicas{world}" if world > 1 else "single"},
        "timing": {"step_ms_median": statistics.median(step_ms), "step_ms_mean":
                   statistics.mean(step_ms), "step_ms_min": min(step_ms),
                   "kernel_ms_mean": statistics.mean(kern_ms),
                   "kernel_ms_median": statistics.median(kern_ms), "wall_s": wall,
                   **({"warm_l2": warm} if warm else {})},
        "roofline": roofline,
        "ffma": ffma,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": input_bytes,
                "d2h_bytes_per_step": 4 * M * N, "steps": e2e_steps, "entry": "gemm_f32_host"},
        "gpu_launches": K_steps * plan["kernels"],
        "clocks": clocks,
        "context": context,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def run_curve(args) -> int:
    """--curve: square sizes 128 .. 8192 for both kernels and cuBLAS context, as CSV.

    The scaling report of "Lecture 12: final project" (its roofline report
    program, CSV columns kernel, size, ms, gflops, bytes_gb, ai, bw_gbs,
    occup, check) on this library: per size and kernel the median call time
    over `--steps` calls (L2 flushed between calls below 256 MiB of inputs),
    TFLOP/s, compulsory bytes 4(MK + KN + MN), arithmetic intensity, the
    bandwidth those bytes imply, the fraction of the kernel's roofline, the
    occupancy of the main kernel (resident threads per SM over the SM's
    maximum, from the occupancy calculator through the library's plan; empty
    for cuBLAS), and the check of the output against the CPU oracle within
    1e-3 + 1e-3 |ref| after the timing: every output up to 2048, beyond that
    the first and last rows and columns plus 4096 random entries (the oracle
    evaluates those one by one).  `checked` is the number of outputs compared.
    """
    import numpy as np
    import torch

    import dense_fp32_gemm_row_gb300 as g
    import oracle
    from seeded_inputs import make_workload

    g.load()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    peaks, _ = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    max_threads = int(getattr(props, "max_threads_per_multi_processor", 2048) or 2048)
    mhz = float(peaks.get("sm_max_mhz") or 2070.0)
    peak_ffma = props.multi_processor_count * FFMA_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
    peak_3x = float(peaks.get("bf16_tflops", 1900.0)) * NOMINAL_TF32_TFLOPS / NOMINAL_BF16_TFLOPS / 3
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    print("kernel,size,ms,tflops,bytes_gb,ai,bw_gbs,pct_roofline,occup,check,checked", flush=True)
    sizes = [int(x) for x in args.curve_sizes.split(",")]
    for n in sizes:
        A_np, B_np = make_workload(2, M=n, N=n, K=n)
        a = torch.from_numpy(A_np).to(dev)
        b = torch.from_numpy(B_np).to(dev)
        c = torch.empty((n, n), dtype=torch.float32, device=dev)
        big = 8 * n * n >= 256 * 1024 * 1024
        # the oracle's values: the whole product up to 2048, else edge rows
        # and columns and random entries
        if n <= 2048:
            rows = cols = None
            want = oracle.ref_gemm(A_np, B_np)
        else:
            rng = np.random.default_rng(n)
            ar = np.arange(n)
            rows = np.concatenate([np.zeros(n, np.int64), np.full(n, n - 1), ar, ar,
                                   rng.integers(0, n, 4096)])
            cols = np.concatenate([ar, ar, np.zeros(n, np.int64), np.full(n, n - 1),
                                   rng.integers(0, n, 4096)])
            want = oracle.ref_gemm_entries(A_np, B_np, rows, cols)
        flops = 2.0 * n ** 3
        bytes_ = 4.0 * 3 * n * n
        for name in ("ffma", "3xtf32", "cublas"):
            occup = ""
            if name == "cublas":
                prev = torch.backends.cuda.matmul.allow_tf32
                torch.backends.cuda.matmul.allow_tf32 = False

                def call():
                    torch.matmul(a, b, out=c)
            else:
                algo = g.ALGOS[name]
                st, plan = g.gemm_f32_plan(n, n, n, algo, 0, a.data_ptr(), b.data_ptr(),
                                           c.data_ptr())
                g.check(st, "gemm_f32_plan")
                occup = f"{plan['ctas_per_sm'] * plan['threads_per_cta'] / max_threads:.3f}"

                def call():
                    g.check(g.gemm_f32_algo(a.data_ptr(), b.data_ptr(), c.data_ptr(), n, n, n,
                                            algo, stream.cuda_stream), name)
            for _ in range(3):
                call()
            times = []
            for _ in range(args.steps):
                if not big:
                    flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            if name == "cublas":
                torch.backends.cuda.matmul.allow_tf32 = prev
            ms = statistics.median(times)
            tf = flops / (ms * 1e-3) / 1e12
            got = c.cpu().numpy()
            got = got if rows is None else got[rows, cols]
            ok = oracle.compare(got, want)["pass"]
            peak = {"ffma": peak_ffma, "3xtf32": peak_3x, "cublas": peak_ffma}[name]
            print(f"{name},{n},{ms:.4f},{tf:.2f},{bytes_ / 1e9:.4f},{flops / bytes_:.1f},"
                  f"{bytes_ / (ms * 1e-3) / 1e9:.1f},{100 * tf / peak:.1f},{occup},"
                  f"{'pass' if ok else 'FAIL'},{got.size}", flush=True)
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description="FP32 GEMM benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", choices=["auto", "ffma", "3xtf32"], default="auto")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--workload", default="square_8192_normal")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-context", action="store_true", help="skip the cuBLAS context timing")
    ap.add_argument("--no-ffma", action="store_true",
                    help="skip the CUDA-core kernel's timing after the timed region")
    ap.add_argument("--ffma-steps", type=int, default=10)
    ap.add_argument("--curve", action="store_true",
                    help="print the size-scaling CSV (128 .. 8192) instead of the JSON line")
    ap.add_argument("--curve-sizes", default="128,256,512,1024,2048,4096,8192")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.curve:
        return run_curve(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
