#!/usr/bin/env python3
"""Benchmark of the GEMM hot path on one GB300.

Metric: GEMM TFLOP/s at M = N = K = 8192, BF16 inputs U[-1,1], FP32
accumulation, BF16 output, device-timed with CUDA events, and its fraction of
the dense BF16 tensor peak.  One step = one gemm_bf16 call through the C ABI
on that workload (host validation, planning, descriptors, the persistent
CTA-pair kernel).  The inputs (256 MiB of A and B) are larger than the 129 MB
L2, so no flush is needed between timed iterations.

Prints ONE JSON line.  Flags: --gpus N --steps K --warmup W
[--impl reference] [--no-variants] [--no-cpu-baseline].

The library runs on one GPU only: its multicast kernel may read only the
memory of the GPU it runs on, and no part of it exchanges data between GPUs.
So this benchmark refuses --gpus above 1 and any launch with WORLD_SIZE above
1 (status 2, before any GPU work).

After the K timed steps the same launch runs back to back for at least two
seconds (the "sustained" object: the GPU settles at its power cap there, so
that figure is compared with the sustained peak).  The other method workloads
follow as "variants", each with its own oracle timing on the host cores.

--impl reference times the CPU oracle (FP64 triple loop, test infrastructure)
on a bounded sample of rows of the same product, on this machine's host cores
(rank 0 only under a multi-rank launcher; the other ranks exit without work).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "GEMM TFLOPS at 8192^3 BF16 (device-timed) and % of dense BF16 tensor peak"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_gemm_8192.txt")
# Sources of the benchmark's kernel (the dense two-consumer pair kernel and
# the host code that launches it): the committed DRAM traffic figure is
# reported only while their code-only hash matches the one it was taken on.
KERNEL_SOURCES = ["gemm_tc.cu", "ptx.cuh", "layout.h", "params.h", "api.cu"]
KERNEL_NAMES = {2: "persistent 1-CTA", 3: "persistent CTA pair (cta_group::2)",
                4: "swapped small-M", 5: "two pairs sharing B by TMA multicast",
                6: "persistent CTA pair, two MMA consumers (cta_group::2)"}
ONE_GPU = ("one GPU only: the library's kernels run on a single GPU (its multicast loads may read "
           "only that GPU's memory) and it has no multi-GPU path")
SUSTAINED_S = 2.2
# The workload, identical in both arms' lines.
CONFIG = {"workload": "gemm_8192x8192x8192_bf16in_fp32acc_bf16out", "M": 8192, "N": 8192, "K": 8192,
          "inputs": "U[-1,1], seed 1003, row-major A and B",
          "layout": "A [M,K] and B [K,N] row-major, D [M,N] row-major",
          "l2": "inputs larger than L2 (A+B = 256 MiB > 129 MB); no flush",
          "parallelism": "single GPU"}


# ----------------------------------------------------------------- infra ----

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    return rank, world


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
            return
        # nvidia-smi's first query initialises NVML, which can hold up CUDA
        # launches from this process for seconds: wait for its first sample
        # so that the set-up does not fall inside the timed region.
        t0 = time.monotonic()
        while time.monotonic() - t0 < 20.0 and self.proc.poll() is None:
            self.out.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sms, maxes, power, reasons = [], [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != len(self.FIELDS):
                    continue
                try:
                    sms.append(float(parts[0]))
                    maxes.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.REASONS, parts[4:]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_max": max(power) if power else None}


def kernel_source_hash(read=None) -> str:
    """Code-only hash of the benchmark kernel's sources (KERNEL_SOURCES)."""
    import hashlib
    from blackwell_tensor_core_gb300 import build
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        if read is None:
            with open(os.path.join(build.CSRC, name), encoding="utf-8") as f:
                text = f.read()
        else:
            text = read(name)
        h.update(build.code_only(text).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256_16") != kernel_source_hash():
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------- timing -------

def time_launches(launch, steps, stream, between=None, keep_ahead=False):
    """Times `steps` launches on `stream`.  Returns (total_ms, per-launch ms list).
    keep_ahead: a GPU sleep before the first timed launch lets the host queue
    the launches ahead of the GPU, so that short kernels are timed without
    host gaps (the sleep lies outside every timed interval)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if keep_ahead:
        torch.cuda._sleep(min(2_000_000 + 20_000 * steps, 40_000_000))
    t0.record(stream)
    for i in range(steps):
        if between is not None:
            between(i)
        starts[i].record(stream)
        launch(i)
        ends[i].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1), [s.elapsed_time(e) for s, e in zip(starts, ends)]


def launch_stats(per, window=20):
    """Median, min and max of per-launch times (ms), and the lowest and
    highest mean over `window` consecutive launches (the MegaMoE page's
    windowed average of back-to-back launches)."""
    out = {"median": statistics.median(per), "min": min(per), "max": max(per), "launches": len(per)}
    if len(per) >= window:
        sums = [math.fsum(per[i:i + window]) for i in range(len(per) - window + 1)]
        out["window_mean_%d" % window] = {"min": min(sums) / window, "max": max(sums) / window}
    return out


def toolchain():
    """nvcc and torch versions the library was built and run with."""
    import torch
    from blackwell_tensor_core_gb300 import build
    try:
        r = subprocess.run([build.nvcc(), "--version"], capture_output=True, text=True, timeout=30)
        nv = [ln for ln in r.stdout.splitlines() if "release" in ln][-1].strip()
    except (OSError, IndexError, RuntimeError, subprocess.SubprocessError):
        nv = "unknown"
    return {"nvcc": nv, "torch": torch.__version__, "arch": "sm_103a"}


def dense_launcher(ops, A, B, D, out_code, stream):
    """launch(i) -> one gemm_bf16 call.  A and B may be lists of equally
    shaped input sets, taken in turn (rotating buffers)."""
    As = A if isinstance(A, (list, tuple)) else [A]
    Bs = B if isinstance(B, (list, tuple)) else [B]
    M, K = As[0].shape
    N = Bs[0].shape[1]
    ptrs = [(a.data_ptr(), b.data_ptr()) for a, b in zip(As, Bs)]
    d, h = D.data_ptr(), stream.cuda_stream

    def launch(i=0):
        a, b = ptrs[i % len(ptrs)]
        ops.gemm_bf16(a, b, d, M, N, K, K, N, N, out_code, h)
    return launch


def check_device_error(ops):
    st, word = ops.last_device_error()
    if st != 0:
        raise RuntimeError("device error word %#x (status %d)" % (word, st))


# ------------------------------------------------------------ oracle --------

def oracle_rate(A_bits, B_bits, budget_s, max_rows=None, threads=None, what=""):
    """The oracle as it stands, on blocks of rows of A x B in order, until
    about `budget_s` seconds of work (or `max_rows` rows).  Returns the
    cpu_baseline object (TFLOP/s over the rows done, 2 * rows * N * K)."""
    import oracle
    oracle.build()
    all_threads = oracle.num_threads()
    if threads is not None:
        oracle.set_num_threads(threads)
    try:
        cores = oracle.num_threads()
        M, K = A_bits.shape
        N = B_bits.shape[1]
        limit = M if max_rows is None else min(M, max_rows)
        oracle.gemm(A_bits, B_bits, rows=(0, min(2, limit)))  # load the library, touch the inputs
        block = max(1, min(limit, 2 * cores))
        rows, dt = 0, 0.0
        while dt < budget_s and rows < limit:
            n = min(block, limit - rows)
            t0 = time.perf_counter()
            oracle.gemm(A_bits, B_bits, rows=(rows, rows + n))
            dt += time.perf_counter() - t0
            rows += n
    finally:
        oracle.set_num_threads(all_threads)
    return {"value": 2.0 * rows * N * K / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": "%s%d of %d rows of the %dx%dx%d product (%d outputs), FP64, %.1f s"
                      % (what, rows, M, M, N, K, rows * N, dt)}


def cpu_baseline(case, budget_s=12.0):
    """The oracle on a bounded row sample of the benchmark product."""
    from blackwell_tensor_core_gb300 import workloads as wl
    return oracle_rate(wl.bits(case.A), wl.bits(case.B), budget_s)


def run_reference(args):
    """Reference arm: the CPU oracle on a bounded sample per step."""
    import oracle
    from blackwell_tensor_core_gb300 import workloads as wl
    oracle.build()
    case = wl.large_case()
    Ab, Bb = wl.bits(case.A), wl.bits(case.B)

    def rows_once(rows, start):
        t0 = time.perf_counter()
        oracle.gemm(Ab, Bb, rows=(start, start + rows))
        return time.perf_counter() - t0

    per_row = rows_once(2, 0) / 2
    rows = max(1, int(120.0 / max((args.steps + args.warmup) * per_row, 1e-9)))
    rows = min(rows, case.M)
    for i in range(args.warmup):
        rows_once(rows, (i * rows) % (case.M - rows + 1))
    times = [rows_once(rows, ((args.warmup + i) * rows) % (case.M - rows + 1)) for i in range(args.steps)]
    value = 2.0 * rows * case.N * case.K * len(times) / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": dict(CONFIG),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": "%d rows of the 8192^3 product per step (%d outputs, K=8192), "
                                   "FP64 triple loop" % (rows, rows * case.N)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------- variants -------

def measure_variants(ops, wl, stream, peaks, steps, only=None, warm=5):
    """Shorter measurements of the other method workloads (same JSON line)."""
    import torch
    out = {}
    dev = torch.device("cuda")
    if only in (None, "tile"):
        out.update(_variant_tile(ops, wl, stream, steps, warm, dev))
    if only in (None, "small_m"):
        out.update(_variant_small_m(ops, wl, stream, peaks, steps, warm, dev))
    if only in (None, "square"):
        out.update(_variant_square(ops, wl, stream, peaks, steps, warm, dev))
    if only in (None, "large_cold"):
        out.update(_variant_large_cold(ops, wl, stream, peaks, steps, warm, dev))
    if only in (None, "grouped"):
        out.update(_variant_grouped(ops, wl, stream, peaks, steps, warm, dev))
    return out


def _variant_tile(ops, wl, stream, steps, warm, dev):
    """The one-tile integer case (256x256x512, FP32 out): a latency figure."""
    import torch
    c = wl.tile_case()
    A, B = c.A.to(dev), c.B.to(dev)
    D = torch.empty((c.M, c.N), dtype=torch.float32, device=dev)
    launch = dense_launcher(ops, A, B, D, wl.OUT_FP32, stream)
    for _ in range(warm):
        launch()
    _, per = time_launches(launch, steps, stream, keep_ahead=True)
    check_device_error(ops)
    return {"tile_256x256x512_fp32out": {"ms_per_launch_median": statistics.median(per),
                                         "ms_per_launch_min": min(per),
                                         "note": "one CTA pair; launch latency dominates"}}


def cublas_context(ops, stream, dev, reps=40):
    """torch.matmul (cuBLAS) on the benchmark workload, launches alternated
    with ours in blocks of 10, medians of CUDA-event times: context for the
    roofline fraction, not part of the measured path."""
    import torch
    from blackwell_tensor_core_gb300 import workloads as wl
    c = wl.large_case()
    A, B = c.A.to(dev), c.B.to(dev)
    D = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    D2 = torch.empty_like(D)
    ours = dense_launcher(ops, A, B, D, wl.OUT_BF16, stream)
    theirs = lambda i=0: torch.matmul(A, B, out=D2)  # noqa: E731
    mo, mc, n = alternate_with_cublas(ops, ours, theirs, stream, reps)
    return {"ours_ms_median": mo, "cublas_ms_median": mc, "ours_tflops": c.flops / (mo * 1e-3) / 1e12,
            "cublas_tflops": c.flops / (mc * 1e-3) / 1e12, "ours_over_cublas": mc / mo,
            "launches_each": n}


def alternate_with_cublas(ops, ours, theirs, stream, reps, between=None):
    """Medians (ms) of CUDA-event times of `ours` and `theirs`, launched
    alternately in blocks of 10 after three untimed launches of each;
    `between` (e.g. an L2 flush) runs before every timed launch of both."""
    for _ in range(3):
        ours()
        theirs()
    to, tc = [], []
    for _ in range(reps // 10):
        to += time_launches(ours, 10, stream, between=between, keep_ahead=True)[1]
        tc += time_launches(theirs, 10, stream, between=between, keep_ahead=True)[1]
    check_device_error(ops)
    return statistics.median(to), statistics.median(tc), len(to)


def _variant_small_m(ops, wl, stream, peaks, steps, warm, dev):
    import torch
    out = {}
    # small-M swapped kernel: HBM-bound, report algorithmic GB/s
    c = wl.small_m_case()
    A, B = c.A.to(dev), c.B.to(dev)
    D = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    launch = dense_launcher(ops, A, B, D, wl.OUT_BF16, stream)
    for _ in range(warm):
        launch()
    _, per = time_launches(launch, steps, stream, keep_ahead=True)
    check_device_error(ops)
    ms = statistics.mean(per)
    nbytes = 2 * (c.M * c.K + c.K * c.N + c.M * c.N)
    gbs = nbytes / (ms * 1e-3) / 1e9
    v = {"ms_per_launch": ms, "tflops": c.flops / (ms * 1e-3) / 1e12, "launch_ms": launch_stats(per),
         "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                      "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes},
         "l2": "B (235 MB) larger than L2"}
    # context: torch.matmul (cuBLAS) on the same inputs, alternated
    D2 = torch.empty_like(D)
    mo, mc, n = alternate_with_cublas(ops, launch, lambda i=0: torch.matmul(A, B, out=D2), stream, 40)
    v["context_cublas"] = {"ours_ms_median": mo, "cublas_ms_median": mc, "ours_over_cublas": mc / mo,
                           "launches_each": n}
    out["small_m_72x16384x7168"] = v
    return out


def _variant_square(ops, wl, stream, peaks, steps, warm, dev):
    import torch
    out = {}
    # square 4096: inputs fit in L2, so flush L2 between timed launches
    c = wl.square_case()
    A, B = c.A.to(dev), c.B.to(dev)
    D = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    launch = dense_launcher(ops, A, B, D, wl.OUT_BF16, stream)
    for _ in range(warm):
        launch()
    _, per = time_launches(launch, steps, stream, between=lambda i: flush.zero_())
    check_device_error(ops)
    ms = statistics.mean(per)
    tf = c.flops / (ms * 1e-3) / 1e12
    out["square_4096"] = {"ms_per_launch": ms, "tflops": tf, "launch_ms": launch_stats(per),
                          "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                                       "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"]},
                          "l2": "flushed (256 MiB write) before every timed launch"}
    # context: torch.matmul (cuBLAS) on the same inputs, alternated, the
    # same flush before every timed launch of either
    D2 = torch.empty_like(D)
    mo, mc, n = alternate_with_cublas(ops, launch, lambda i=0: torch.matmul(A, B, out=D2), stream, 40,
                                      between=lambda i: flush.zero_())
    out["square_4096"]["context_cublas"] = {"ours_ms_median": mo, "cublas_ms_median": mc,
                                            "ours_over_cublas": mc / mo, "launches_each": n}
    return out


def _variant_large_cold(ops, wl, stream, peaks, steps, warm, dev):
    """The benchmark product on two rotating input sets (512 MiB of A and B),
    so that no launch finds its inputs in L2 from the launch before."""
    import torch
    c = wl.large_case()
    c2 = wl.large_case(seed=2003)
    As = [c.A.to(dev), c2.A.to(dev)]
    Bs = [c.B.to(dev), c2.B.to(dev)]
    D = torch.empty((c.M, c.N), dtype=torch.bfloat16, device=dev)
    launch = dense_launcher(ops, As, Bs, D, wl.OUT_BF16, stream)
    for i in range(warm):
        launch(i)
    _, per = time_launches(launch, steps, stream)
    check_device_error(ops)
    ms = statistics.mean(per)
    tf = c.flops / (ms * 1e-3) / 1e12
    return {"large_8192_rotating": {
        "ms_per_launch": ms, "tflops": tf, "launch_ms": launch_stats(per),
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / peaks["bf16_tflops"]},
        "l2": "two input sets (2 x 256 MiB) taken in turn: cold L2 for every launch"}}


def _variant_grouped(ops, wl, stream, peaks, steps, warm, dev):
    """Grouped expert FC1, FC1 + SwiGLU and FC2, launched in alternating blocks
    of ten so that the three see the same clocks (after the long 8192^3 loop
    the GPU runs at its power cap, and the clock drifts as it warms); then
    FC1 on two rotating input sets."""
    import torch
    out = {}
    c = wl.grouped_case()
    A = c.A.to(dev)
    Bs = [b.to(dev) for b in c.Bs]
    off = torch.from_numpy(c.offsets).to(dev)
    D = torch.empty((c.total, c.N), dtype=torch.bfloat16, device=dev)
    H = torch.empty((c.total, c.N // 2), dtype=torch.bfloat16, device=dev)  # B_g = [gate | up]
    bptrs = [b.data_ptr() for b in Bs]
    a, d, hp, o, h = A.data_ptr(), D.data_ptr(), H.data_ptr(), off.data_ptr(), stream.cuda_stream
    # expert FC2 (down projection) over the same buckets: K = 2048, N = 4096
    c2 = wl.grouped_fc2_case()
    A2 = c2.A.to(dev)
    B2 = [b.to(dev) for b in c2.Bs]
    D2 = torch.empty((c2.total, c2.N), dtype=torch.bfloat16, device=dev)
    b2ptrs = [b.data_ptr() for b in B2]
    a2, d2 = A2.data_ptr(), D2.data_ptr()
    launches = {
        "grouped_fc1_32x4096x4096": (
            lambda i=0: ops.grouped_gemm_bf16(a, bptrs, d, o, c.G, c.total, c.N, c.K, h),
            c.flops, {"rows": c.total, "l2": "A + B (1.34 GB) larger than L2"}),
        "grouped_fc1_swiglu_32x4096x4096": (
            lambda i=0: ops.grouped_gemm_swiglu_bf16(a, bptrs, hp, o, c.G, c.total, c.N, c.K, h), c.flops,
            {"rows": c.total, "out_cols": c.N // 2, "l2": "A + B (1.34 GB) larger than L2"}),
        "grouped_fc2_32x4096x2048": (
            lambda i=0: ops.grouped_gemm_bf16(a2, b2ptrs, d2, o, c2.G, c2.total, c2.N, c2.K, h),
            c2.flops, {"rows": c2.total, "l2": "A + B (0.67 GB) larger than L2"}),
    }
    for fn, _, _ in launches.values():
        for _ in range(warm):
            fn()
    per = {k: [] for k in launches}
    blocks = max(1, max(10, steps // 4) // 10)
    for _ in range(blocks):
        for k, (fn, _, _) in launches.items():
            fn()  # one untimed launch after each switch of workload
            per[k] += time_launches(fn, 10, stream)[1]
    check_device_error(ops)
    for k, (_, flops, extra) in launches.items():
        ms = statistics.mean(per[k])
        tf = flops / (ms * 1e-3) / 1e12
        out[k] = dict({"ms_per_launch": ms, "tflops": tf,
                       "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                                    "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"]}}, **extra)
        out[k]["launch_ms"] = launch_stats(per[k])
    del A2, B2, D2, H
    # rotating inputs: a second FC1 input set (activations and weights)
    c3 = wl.grouped_case(seed=2005)
    A3 = c3.A.to(dev)
    B3 = [b.to(dev) for b in c3.Bs]
    off3 = torch.from_numpy(c3.offsets).to(dev)
    sets = [(a, bptrs, o), (A3.data_ptr(), [b.data_ptr() for b in B3], off3.data_ptr())]

    def fc1_rot(i=0):
        ai, bi, oi = sets[i % 2]
        ops.grouped_gemm_bf16(ai, bi, d, oi, c.G, c.total, c.N, c.K, h)
    for i in range(warm):
        fc1_rot(i)
    _, per_rot = time_launches(fc1_rot, max(10, steps // 2), stream)
    check_device_error(ops)
    ms = statistics.mean(per_rot)
    tf = c.flops / (ms * 1e-3) / 1e12
    out["grouped_fc1_32x4096x4096_rotating"] = {
        "ms_per_launch": ms, "tflops": tf, "launch_ms": launch_stats(per_rot),
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / peaks["bf16_tflops"]},
        "l2": "two input sets (2 x 1.34 GB, each with its own routing counts) taken in turn"}
    return out


def run_only(args):
    """Profiling aid: one variant workload on its own (warm-up + steps)."""
    import torch
    from blackwell_tensor_core_gb300 import build, ops
    from blackwell_tensor_core_gb300 import workloads as wl
    build.build()
    peaks, _ = load_peaks()
    stream = torch.cuda.current_stream()
    res = measure_variants(ops, wl, stream, peaks, args.steps, only=args.only, warm=args.warmup)
    print(json.dumps(res), flush=True)


# --------------------------------------------------------------- ours -------

def sustained_window(ops, launch, flops, stream, peaks, ms_hint):
    """At least SUSTAINED_S seconds of back-to-back launches, with the clocks
    sampled over them: the GPU reaches its power cap here."""
    import torch
    n = max(200, int(math.ceil(SUSTAINED_S * 1e3 / max(ms_hint, 1e-3))))
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(3):
        launch()
    total_ms, per = time_launches(launch, n, stream)
    clocks = sampler.stop()
    check_device_error(ops)
    ms = total_ms / n
    tf = flops / (ms * 1e-3) / 1e12
    return {"launches": n, "region_ms": total_ms, "ms_per_launch": ms, "tflops": tf,
            "peak_sustained": peaks["bf16_tflops_sustained"],
            "frac_of_sustained_peak": tf / peaks["bf16_tflops_sustained"],
            "frac_of_burst_peak": tf / peaks["bf16_tflops"],
            "launch_ms": dict(launch_stats(per), first_tenth_mean=statistics.mean(per[:n // 10]),
                              last_tenth_mean=statistics.mean(per[-(n // 10):])),
            "clocks": clocks}


def run_ours(args):
    import torch
    from blackwell_tensor_core_gb300 import build, ops
    from blackwell_tensor_core_gb300 import workloads as wl

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device (there is no CPU path)")
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    build.build()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    case = wl.large_case() if args.size is None else wl.large_case(n=args.size)
    A, B = case.A.to(dev), case.B.to(dev)
    D = torch.empty((case.M, case.N), dtype=torch.bfloat16, device=dev)
    launch = dense_launcher(ops, A, B, D, wl.OUT_BF16, stream)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    check_device_error(ops)

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(3):  # keep the clocks up after the sampler's start-up
        launch()
    total_ms, per = time_launches(launch, args.steps, stream)
    clocks = sampler.stop()
    check_device_error(ops)

    flops = case.flops
    value = flops * args.steps / (total_ms * 1e-3) / 1e12
    mean_launch = statistics.mean(per)
    achieved = flops / (mean_launch * 1e-3) / 1e12
    # A timed region of a few hundred milliseconds runs before the power cap
    # bites: compare it with the burst peak.  Seconds-long regions settle at
    # the power-capped clock: compare those with the sustained peak.
    long_region = total_ms >= 2000.0
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak = peaks[peak_key]
    traffic = recorded_traffic()
    plan = ops.plan(case.M, case.N, case.K, sm_count=torch.cuda.get_device_properties(dev).multi_processor_count)

    sustained = None
    if not args.no_sustained:
        sustained = sustained_window(ops, launch, flops, stream, peaks, mean_launch)

    # end to end through the host-buffer entry point (copies in the timed region)
    hA, hB = case.A.pin_memory(), case.B.pin_memory()
    hD = torch.empty((case.M, case.N), dtype=torch.bfloat16).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))

    def e2e_launch(i=0):
        ops.gemm_bf16_host(hA, hB, hD, A, B, D, stream)
    e2e_launch()
    torch.cuda.synchronize()
    e2e_ms, _ = time_launches(e2e_launch, e2e_steps, stream)
    check_device_error(ops)
    e2e = {"value": flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": 2 * case.M * case.K + 2 * case.K * case.N,
           "d2h_bytes_per_step": 2 * case.M * case.N, "steps": e2e_steps,
           "api": "gemm_bf16_host (pinned host buffers, H2D + GEMM + D2H on one stream)"}
    del hA, hB, hD

    variants = None
    variant_clocks = None
    if not args.no_variants:
        vs = ClockSampler(torch.cuda.current_device())
        vs.start()
        variants = measure_variants(ops, wl, stream, peaks, min(args.steps, 200))
        variant_clocks = vs.stop()
        # the variants run right after the long timed loop, at the power cap:
        # give their fractions of the sustained figure too
        for v in variants.values():
            r = v.get("roofline")
            if r and r.get("unit") == "TFLOP/s":
                r["frac_of_sustained"] = r["achieved"] / peaks["bf16_tflops_sustained"]

    context = None
    if not args.no_variants:
        context = cublas_context(ops, stream, dev)

    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(case)
        if variants is not None:
            # the oracle on each variant's own product (host cores only)
            for name, v in measure_variant_oracles(wl).items():
                if name in variants:
                    variants[name].update(v)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(CONFIG),
        "build": {"kernel": "%s, tile %dx%dx64, %d stages, grid %d" % (
                      KERNEL_NAMES.get(plan.kernel, plan.kernel), plan.tile_m, plan.tile_n, plan.stages,
                      plan.grid),
                  "cluster": 2, "gpu": torch.cuda.get_device_name(dev), "toolchain": toolchain(),
                  "library": ops.version()},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": "%s %s (timed region %.0f ms)" % (peak_src, peak_key, total_ms),
                     "frac_of_burst_peak": achieved / peaks["bf16_tflops"],
                     "frac_of_sustained_peak": achieved / peaks["bf16_tflops_sustained"],
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": 3 * 2 * case.M * case.N},
        "sustained": sustained,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks,
        "launch_ms": dict(launch_stats(per), mean=mean_launch,
                          first_tenth_mean=statistics.mean(per[:max(1, len(per) // 10)]),
                          last_tenth_mean=statistics.mean(per[-max(1, len(per) // 10):])),
        "variants": variants,
        "variants_clocks": variant_clocks,
        "context_cublas": context,
    }
    print(json.dumps(line), flush=True)


def measure_variant_oracles(wl):
    """cpu_baseline objects of the variant workloads (oracle on host cores;
    bounded samples, a few seconds each)."""
    out = {}
    c = wl.tile_case()
    out["tile_256x256x512_fp32out"] = {"cpu_baseline": oracle_rate(wl.bits(c.A), wl.bits(c.B), 1.0)}
    c = wl.small_m_case()
    out["small_m_72x16384x7168"] = {"cpu_baseline": oracle_rate(wl.bits(c.A), wl.bits(c.B), 10.0)}
    c = wl.square_case()
    Ab, Bb = wl.bits(c.A), wl.bits(c.B)
    out["square_4096"] = {"cpu_baseline": oracle_rate(Ab, Bb, 3.0),
                          "cpu_baseline_one_core": oracle_rate(Ab, Bb, 3.0, threads=1)}
    for name, case in (("grouped_fc1_32x4096x4096", wl.grouped_case()),
                       ("grouped_fc2_32x4096x2048", wl.grouped_fc2_case())):
        # one expert's rows against its own weight: the same arithmetic per row
        g = int(max(range(case.G), key=lambda j: case.offsets[j + 1] - case.offsets[j]))
        r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
        out[name] = {"cpu_baseline": oracle_rate(wl.bits(case.A[r0:r1]), wl.bits(case.Bs[g]), 3.0,
                                                 what="expert %d: " % g)}
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sustained", action="store_true",
                    help="skip the two-second back-to-back window (profiling runs)")
    ap.add_argument("--size", type=int, default=None,
                    help="square size of the timed GEMM (default 8192; smaller only for profiling)")
    ap.add_argument("--only", choices=["tile", "small_m", "square", "large_cold", "grouped"], default=None,
                    help="profiling aid: run only one variant workload, print its numbers")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    rank, world = dist_env()
    if args.impl == "reference":
        # host cores only; under a multi-rank launcher rank 0 alone runs it
        if rank == 0:
            run_reference(args)
        return
    if args.gpus != 1 or world != 1:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "impl": "ours", "n_gpus": max(args.gpus, world),
                              "unavailable": ONE_GPU}), flush=True)
        sys.stderr.write("bench.py: %s\n" % ONE_GPU)
        sys.exit(2)
    if args.only:
        run_only(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
