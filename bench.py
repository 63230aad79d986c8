#!/usr/bin/env python3
"""Throughput of the row-major FP32 GEMM on GB300; prints ONE JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8192x8192x8192]
                    [--mode tc3x|ffma|tc1x] [--impl ours|reference]

A step is one product C = A * B of the named problem (workloads.py) through
the C ABI (one kernel launch).  Inputs are synthetic, seeded, resident in
device memory when the timed region starts; K steps are timed with CUDA
events on the launching stream, bracketed by a barrier and a synchronise.
Problems whose operands fit twice in L2 get an L2 flush between steps
(each step timed on its own); the default 8192^3 problem's operands are
larger than L2.  `value` is whole-job TFLOPS = 2MNK * ranks / max-over-ranks
time.  The e2e figure times gemm_f32_host, the C-ABI call on host buffers:
every step copies A and B in from pinned host memory, computes and copies C
back; consecutive calls overlap one's copies with the next one's product.
The latency of one such call, waited for alone, is reported beside it.

With N > 1 (torchrun) every rank runs its own replica of the problem on its
own GPU: the product needs no exchange between GPUs, so scaling is weak.

--impl reference times the CPU oracle (the only other implementation of the
same computation here) on a bounded sample of the same problem: the first R
rows of A times all of B, R chosen so the run ends within a few minutes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FP32 GEMM TFLOPS (2MNK/t) at 1 GB300 and % of 3xTF32 / FFMA roofline"
L2_BYTES = 129 * 1024 * 1024
# nominal dense ratio (tf32 : bf16 tensor rate): scales the measured bf16
# cuBLAS peak into the secondary tensor roof the line also reports
TF32_PER_BF16 = 1.1 / 2.25
MODE_PRODUCTS = {"tc3x": 3, "tc1x": 1, "ffma": 1}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="8192x8192x8192", choices=sorted(workloads.PROBLEMS))
    ap.add_argument("--mode", default="tc3x", choices=sorted(MODE_PRODUCTS))
    ap.add_argument("--flags", type=lambda s: int(s, 0), default=0, help="gemm_f32_ex flags (tuning)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-sub-modes", action="store_true",
                    help="leave out the ffma and tc1x records timed beside the headline mode")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the one-line benchmark: every problem of workloads.py in every "
                         "mode, warm and cold L2, mean and median, and the pages' statistic (one "
                         "JSON line per row, then a table on stderr)")
    ap.add_argument("--oracle-table", action="store_true",
                    help="instead of the one-line benchmark: time the CPU oracle on every problem "
                         "of workloads.py with all host threads (and with one thread for the small "
                         "ones), the host's core count and CPU model alongside (one JSON line per "
                         "row, then a table on stderr); needs no GPU")
    ap.add_argument("--ladder", action="store_true",
                    help="instead of the one-line benchmark: time the pages' kernels v0..v4, this "
                         "library's modes and torch.matmul on the pages' two sizes (one JSON line per "
                         "row, then a table on stderr)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed plumbing
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def barrier(dist_mod, device=None):
    if dist_mod is not None:
        if device is not None and device.type == "cuda":
            dist_mod.barrier(device_ids=[device.index])
        else:
            dist_mod.barrier()


def max_over_ranks(value: float, dist_mod, device) -> float:
    """Largest value over all ranks (the job ends when its slowest rank does)."""
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Aggregate throughput: every rank did `steps` products; the job took the max time."""
    return flop_per_step * steps * world / max_seconds / 1e12


# ---------------------------------------------------------------- peaks, clocks, traffic
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 10 ms while active,
    each sample with its timestamp, so that the samples of a window (the
    timed steps) can be told from the rest (warm-up)."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, enabled: bool = True, period_ms: int = 10):
        self.index = index
        self.proc = None
        self.enabled = enabled
        self.period_ms = period_ms
        self.lines = []

    def __enter__(self):
        if self.enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                     "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
            time.sleep(0.3)          # the first sample is out before the work starts
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(2.0 * self.period_ms / 1e3)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def samples(self):
        """[(unix time, sm MHz, max sm MHz, [reason flags])]"""
        import datetime
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                when = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((when, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        return rows

    def summary(self, t0=None, t1=None):
        """Median SM clock and throttle reasons over the samples taken in
        [t0, t1] (host wall-clock seconds); over every sample when that window
        holds fewer than 3 (a timed region shorter than a few sample periods),
        which the record says."""
        rows = self.samples()
        if not rows:
            return None
        window = "timed steps"
        if t0 is not None:
            inside = [r for r in rows if t0 <= r[0] <= t1]
            if len(inside) < 3:
                window = "warm-up and timed steps (%d samples inside the timed steps)" % len(inside)
                inside = [r for r in rows if r[0] <= t1]
            rows = inside or rows
        reasons = sorted({self.REASONS[i] for _, _, _, flags in rows for i, v in enumerate(flags)
                          if v == "Active"})
        out = {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
               "reasons": reasons, "samples": len(rows), "window": window,
               "period_ms": self.period_ms}
        if t1 is not None:
            # the wider record: warm-up and timed steps together
            wide = [r for r in self.samples() if r[0] <= t1]
            if wide:
                out["with_warmup"] = {"sm_mhz": statistics.median(r[1] for r in wide),
                                      "min_sm_mhz": min(r[1] for r in wide), "samples": len(wide)}
        return out


# the sources each kernel's device code comes from: its own file and the
# device header (launch.h is host-side interface only)
KERNEL_SOURCES = {
    "tc_pair_kernel": ("tc_pair_gemm.cu", "device_common.cuh"),
    "tc_gemm_kernel": ("tc_gemm.cu", "device_common.cuh"),
    "ffma_gemm_kernel": ("ffma_gemm.cu", "device_common.cuh"),
}


def source_hash(kernel: str) -> str:
    """Hash of the sources `kernel` is built from: a recorded ncu figure is
    used only while they are unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "accelerator_row_major_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, config: str, mode: str):
    """DRAM bytes per launch from a committed ncu capture of the same sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        table = json.load(f)
    rec = table.get("%s/%s/%s" % (kernel, config, mode))
    if not rec or rec.get("source_sha") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- CPU oracle timing
def oracle_sample(A, B, seconds: float):
    """Time the oracle on the first R rows of A; R grows until ~`seconds`."""
    import oracle
    M, K = A.shape
    N = B.shape[1]
    rows = 1
    while True:
        t0 = time.perf_counter()
        oracle.gemm(A[:rows], B)
        dt = time.perf_counter() - t0
        if dt >= seconds / 8 or rows >= M:
            break
        rows = min(M, rows * 4)
    rows = max(1, min(M, int(rows * seconds / max(dt, 1e-6))))
    t0 = time.perf_counter()
    oracle.gemm(A[:rows], B)
    dt = time.perf_counter() - t0
    tflops = workloads.gemm_flops(rows, N, K) / dt / 1e12
    return {"value": tflops, "unit": "TFLOPS", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": "first %d of %d rows of A times all of B (%dx%dx%d), fp64 accumulation plus "
                      "|A||B|, %.1f s" % (rows, M, rows, K, N, dt)}, rows


def host_cpu():
    """(logical cores, CPU model) of this host, from the OS."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                key = key.strip().lower()
                if key in ("model name", "cpu model", "hardware") and val.strip():
                    model = val.strip()
                    break
                if key == "cpu part" and model == "unknown":
                    model = "cpu part " + val.strip()
    except OSError:
        pass
    return os.cpu_count() or 1, model


# problems small enough to time single-threaded as well
ORACLE_ONE_THREAD = ("100x37x70", "100x37x70-int", "1024x512x1024", "1001x513x777")
# problems timed on a row sample (the full product would take minutes)
ORACLE_SAMPLED = ("8192x8192x8192",)


def run_oracle_table(args):
    """Wall time of the oracle on every problem (generation excluded)."""
    import oracle
    cores, model = host_cpu()
    rows_out = []
    for name in workloads.PROBLEMS:
        p = workloads.PROBLEMS[name]
        A, B = workloads.make_inputs(p.M, p.K, p.N, p.law, p.seed)
        for threads in ((0, 1) if name in ORACLE_ONE_THREAD else (0,)):
            used = oracle.max_threads() if threads == 0 else 1
            if name in ORACLE_SAMPLED:
                base, rows = oracle_sample(A, B, args.cpu_seconds)
                tflops, what = base["value"], base["sample"]
                seconds = workloads.gemm_flops(p.M, p.N, p.K) / (tflops * 1e12)
                kind = "projected from the sample"
            else:
                oracle.gemm(A[:1], B, threads)          # page in and load the library
                t0 = time.perf_counter()
                oracle.gemm(A, B, threads)
                seconds = time.perf_counter() - t0
                tflops = workloads.gemm_flops(p.M, p.N, p.K) / seconds / 1e12
                what, kind = "full product", "measured"
            row = {"oracle_table": name, "M": p.M, "K": p.K, "N": p.N, "threads": used,
                   "seconds": seconds, "tflops": tflops, "timing": kind, "what": what,
                   "host_cores": cores, "cpu_model": model}
            rows_out.append(row)
            print(json.dumps(row), flush=True)
    print("host: %d cores, %s" % (cores, model), file=sys.stderr)
    print("%-6s %-22s %7s %12s %10s  %s" % ("config", "M x K x N", "threads", "seconds", "TFLOPS",
                                            "timing"), file=sys.stderr)
    for r in rows_out:
        print("%-6s %-22s %7d %12.4f %10.4f  %s" % (r["oracle_table"], "%dx%dx%d" % (r["M"], r["K"], r["N"]),
                                                   r["threads"], r["seconds"], r["tflops"], r["timing"]),
              file=sys.stderr)
    return 0


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    p = workloads.PROBLEMS[args.config]
    A, B = workloads.make_inputs(p.M, p.K, p.N, p.law, p.seed)
    budget = 150.0 / max(1, args.steps + args.warmup)
    _, rows = oracle_sample(A, B, min(budget, 5.0))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gemm(A[:rows], B)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = workloads.gemm_flops(rows, p.N, p.K) / t / 1e12
    sample = "first %d of %d rows of A times all of B per step (%dx%dx%d)" % (rows, p.M, rows, p.K, p.N)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "%dx%dx%d (M,K,N) fp32 row-major, %s, seed %d" %
                       (p.M, p.K, p.N, p.law, p.seed), "sample_rows": rows},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU timing
def roofline(kernel, mode, flop, work_bytes, t_kernel, rates, clocks, peaks, peak_src):
    """The binding roof of one launch of `kernel`.  Compute roofs are the
    probed per-SM rate of the unit doing the work (gemm_f32_unit_rates: FLOP
    per SM per clock) x SMs x the SM clock the timed launches ran at: the
    kernels' own clock record when the summary has it, else the median
    nvidia-smi sample (under a tensor-core load the SMs run well below the
    clock nvidia-smi reports, so the record is the one that bounds the
    kernel; the roof at the reported clock is kept beside it).  The memory
    roof is the measured copy bandwidth."""
    sms = rates["num_sms"]
    smi_mhz = clocks.get("sm_mhz") if clocks else None
    kernel_mhz = clocks.get("kernel_sm_mhz") if clocks else None
    if kernel_mhz:
        mhz = kernel_mhz
        clock_src = "SM clock of the timed launches, measured in the kernels: clock64 / " \
                    "%globaltimer of CTA 0"
    elif smi_mhz:
        mhz = smi_mhz
        clock_src = "median SM clock sampled over the %s" % clocks["window"]
    else:
        mhz = rates["sm_mhz"]
        clock_src = "SM clock during the unit probe (no clock samples)"
    if mode == "ffma":
        peak = rates["ffma_flop_per_clk_sm"] * sms * mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": flop / t_kernel / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": "probed fma.rn.f32x2 rate %.1f FLOP/clk/SM x %d SMs x %.0f MHz (%s)"
                               % (rates["ffma_flop_per_clk_sm"], sms, mhz, clock_src)}
    else:
        nprod = MODE_PRODUCTS[mode]
        per_clk = rates["tf32_pair_flop_per_clk_sm"] if kernel == "tc_pair_kernel" \
            else rates["tf32_flop_per_clk_sm"]
        peak = per_clk * sms * mhz * 1e6 / 1e12
        hbm = peaks.get("hbm_gbs")
        # the binding roof: the larger of the two lower bounds on the time
        if hbm and work_bytes / (hbm * 1e9) > nprod * flop / (peak * 1e12):
            roof = {"bound": "hbm", "achieved": work_bytes / t_kernel / 1e9, "peak": hbm,
                    "unit": "GB/s",
                    "peak_source": "%s copy bandwidth; achieved = algorithmic bytes "
                                   "4(MK + KN + MN) per launch / time" % peak_src}
        else:
            roof = {"bound": "tensor", "achieved": nprod * flop / t_kernel / 1e12, "peak": peak,
                    "unit": "TFLOP/s",
                    "peak_source": "probed tcgen05 kind::tf32 rate %.0f FLOP/clk/SM (%s) x %d SMs x "
                                   "%.0f MHz (%s); achieved counts the %d tf32 products per fp32 product"
                                   % (per_clk, "SM pairs" if kernel == "tc_pair_kernel" else "one SM",
                                      sms, mhz, clock_src, nprod)}
            bf16 = peaks["bf16_tflops"] * TF32_PER_BF16
            roof["secondary"] = {"peak": bf16, "frac": roof["achieved"] / bf16,
                                 "peak_source": "%s bf16 cuBLAS burst x nominal tf32/bf16 ratio "
                                                "1.1/2.25" % peak_src}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["frac_of"] = "measured"
    if roof["bound"] != "hbm" and kernel_mhz and smi_mhz:
        # the same roof at the clock nvidia-smi reported for the window
        at = roof["peak"] * smi_mhz / kernel_mhz
        roof["at_reported_clock"] = {"sm_mhz": smi_mhz, "peak": at, "frac": roof["achieved"] / at}
    return roof


def time_product(g, A, B, C, M, N, K, mode, flags, stream, steps, warmup, flush, scratch, dist_mod,
                 device, clocks_enabled, local_rank):
    """W warm-up calls, then exactly `steps` timed calls (CUDA events on the
    launching stream, a barrier and a synchronise on both sides), with
    nvidia-smi sampling from before the warm-up to after the timed steps.
    Returns (max-over-ranks ms per step, kernels per call, kernel name,
    clock summary of the timed window)."""
    import torch

    def step():
        rc = g.gemm_f32_ex(A, B, C, M, N, K, mode, flags, stream)
        if rc != 0:
            raise g.GemmError(rc, "gemm_f32_ex")

    events = []
    with ClockSampler(local_rank, enabled=clocks_enabled) as clocks:
        torch.cuda.synchronize(device)
        with torch.cuda.stream(stream):
            for _ in range(max(3, warmup)):
                step()
        launches_per_step = g.gemm_f32_last_launches()
        kernel = g.gemm_f32_last_kernel()
        rc, site = g.gemm_f32_status(stream)
        if rc != 0:
            raise SystemExit("device error word %d after warm-up" % site)
        barrier(dist_mod, device)
        torch.cuda.synchronize(device)
        rec0 = g.gemm_f32_clock_record(stream)
        t_start = time.time()
        with torch.cuda.stream(stream):
            if flush:
                for _ in range(steps):
                    scratch.zero_()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    step()
                    e1.record(stream)
                    events.append((e0, e1))
            else:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(steps):
                    step()
                e1.record(stream)
                events.append((e0, e1))
        torch.cuda.synchronize(device)
        t_end = time.time()
        rec1 = g.gemm_f32_clock_record(stream)
        barrier(dist_mod, device)
    device_ms = sum(a.elapsed_time(b) for a, b in events)
    rc, site = g.gemm_f32_status(stream)
    if rc != 0:
        raise SystemExit("device error word %d in the timed region" % site)
    ms_per_step = max_over_ranks(device_ms / steps, dist_mod, device)
    return ms_per_step, launches_per_step, kernel, with_kernel_clock(clocks.summary(t_start, t_end),
                                                                     rec0, rec1)


def with_kernel_clock(summary, rec0, rec1):
    """The clock summary with the SM clock the timed launches ran at, from
    the kernels' own clock record (gemm_f32_clock_record read before and
    after them): SM clocks / nanoseconds of CTA 0 over those launches."""
    cycles, ns = rec1[0] - rec0[0], rec1[1] - rec0[1]
    if ns <= 0 or cycles <= 0:
        return summary
    out = dict(summary) if summary else {}
    out["kernel_sm_mhz"] = 1e3 * cycles / ns
    out["kernel_clock"] = ("clock64 / %globaltimer of CTA 0 of each timed launch, summed "
                           "(gemm_f32_clock_record)")
    return out


# modes reported beside the headline one, on the same problem, when the
# default problem is benchmarked (each with its own roof and clocks)
SUB_MODES = ("ffma", "tc1x")


def run_ours(args):
    import numpy as np  # noqa: F401
    import torch

    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist_mod = init_dist(world, "nccl")

    from accelerator_row_major_gb300 import build as build_mod
    build_mod.build()
    import accelerator_row_major_gb300 as g

    p = workloads.PROBLEMS[args.config]
    M, K, N = p.M, p.K, p.N
    A_h, B_h = workloads.make_inputs(M, K, N, p.law, p.seed)
    stream = torch.cuda.Stream(device)
    A = torch.from_numpy(A_h).to(device)
    B = torch.from_numpy(B_h).to(device)
    C = torch.empty((M, N), dtype=torch.float32, device=device)
    flop = workloads.gemm_flops(M, N, K)
    work_bytes = workloads.algorithmic_bytes(M, N, K)
    flush = work_bytes < 2 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device) if flush else None
    rates = g.gemm_f32_unit_rates()        # per-SM unit rates: the compute roofs

    ms_per_step, launches_per_step, kernel, clocks = time_product(
        g, A, B, C, M, N, K, args.mode, args.flags, stream, args.steps, args.warmup, flush, scratch,
        dist_mod, device, not args.no_clocks, local_rank)
    value = whole_job_tflops(flop, args.steps, world, ms_per_step * args.steps / 1e3)

    # ---- the other modes on the same problem, each timed the same way
    subs = {}
    if not args.no_sub_modes and args.flags == 0:
        for mode in SUB_MODES:
            if mode == args.mode:
                continue
            ms, launches, kern, clk = time_product(
                g, A, B, C, M, N, K, mode, 0, stream, args.steps, args.warmup, flush, scratch,
                dist_mod, device, not args.no_clocks, local_rank)
            subs[mode] = {"value": whole_job_tflops(flop, args.steps, world, ms * args.steps / 1e3),
                          "unit": "TFLOPS", "ms_per_step": ms, "steps": args.steps,
                          "warmup": args.warmup, "kernel": kern,
                          "gpu_launches": launches * args.steps, "clocks": clk,
                          "roofline": None, "_t": ms / 1e3}

    # ---- end to end through the C-ABI call with host buffers
    e2e = None
    if not args.no_e2e:
        A_pin = torch.from_numpy(A_h).pin_memory()
        B_pin = torch.from_numpy(B_h).pin_memory()
        C_pin = torch.empty((M, N), dtype=torch.float32).pin_memory()
        # as many queued calls as timed steps: the first call's copy-in and
        # the last one's copy-out are the only copies no product hides (the
        # host link moves ~208 GB/s in and ~191 GB/s out, ~304 GB/s both ways)
        e2e_steps = max(8, args.steps)

        def e2e_call():
            # copies A and B in, computes, copies C out (gemm_f32_host)
            rc = g.gemm_f32_host(A_pin, B_pin, C_pin, M, N, K, args.mode, stream)
            if rc != 0:
                raise g.GemmError(rc, "gemm_f32_host")

        for _ in range(2):          # both device slots allocated before timing
            e2e_call()
        torch.cuda.synchronize(device)
        barrier(dist_mod, device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_call()
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier(dist_mod, device)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist_mod, device)
        # the same call waited for one at a time: one product's latency
        serial = []
        for _ in range(3):
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            e2e_call()
            s1.record(stream)
            s1.synchronize()
            serial.append(s0.elapsed_time(s1))
        serial_ms = max_over_ranks(statistics.median(serial), dist_mod, device)
        e2e = {"value": whole_job_tflops(flop, 1, world, e2e_ms / 1e3), "unit": "TFLOPS",
               "h2d_bytes_per_step": 4 * (M * K + K * N), "d2h_bytes_per_step": 4 * M * N,
               "steps": e2e_steps, "ms_per_step": e2e_ms,
               "call": "gemm_f32_host (C ABI) on pinned host buffers, mode %s" % args.mode,
               "schedule": "calls queued back to back; each copies its A and B in and its C out, "
                           "and one call's copies overlap its neighbour's product (two device "
                           "slots, three streams)",
               "serial_ms_per_step": serial_ms,
               "serial_value": whole_job_tflops(flop, 1, world, serial_ms / 1e3)}
        rc, site = g.gemm_f32_status(stream)
        if rc != 0:
            raise SystemExit("device error word %d in the e2e region" % site)

    if rank != 0:
        if dist_mod is not None:
            dist_mod.destroy_process_group()
        return 0

    peaks, peak_src = measured_peaks()
    roof = roofline(kernel, args.mode, flop, work_bytes, ms_per_step / 1e3, rates, clocks, peaks,
                    peak_src)   # one launch per step
    roof["kernel"] = kernel
    roof["traffic"] = recorded_traffic(kernel, args.config, args.mode)
    roof["algorithmic_bytes"] = work_bytes
    for mode, sub in subs.items():
        sub["roofline"] = roofline(sub["kernel"], mode, flop, work_bytes, sub.pop("_t"), rates,
                                   sub["clocks"], peaks, peak_src)
        sub["roofline"]["traffic"] = recorded_traffic(sub["kernel"], args.config, mode)

    line = {"metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "%dx%dx%d (M,K,N) fp32 row-major, %s, seed %d" %
                       (M, K, N, p.law, p.seed), "M": M, "K": K, "N": N, "mode": args.mode,
                       "flags": args.flags,
                       "l2": "flushed between steps" if flush else "inputs larger than L2",
                       "parallelism": "replicas x%d" % world},
            "roofline": roof, "gpu_launches": launches_per_step * args.steps,
            "unit_rates": rates}
    if e2e is not None:
        line["e2e"] = e2e
    if clocks is not None:
        line["clocks"] = clocks
    for mode, sub in subs.items():
        line[mode] = sub
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(A_h, B_h, args.cpu_seconds)[0]
    print(json.dumps(line), flush=True)
    if dist_mod is not None:
        dist_mod.destroy_process_group()
    return 0


# ---------------------------------------------------------------- the pages' ladder
def time_calls(fn, stream, warmup: int, reps: int, batches: int = 5):
    """Mean device time per call (ms) of `batches` batches of `reps` calls of
    fn() on `stream`, each batch bracketed by CUDA events; warm L2 as on the
    pages (the same inputs every call)."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
    torch.cuda.synchronize()
    means = []
    for _ in range(batches):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        e1.synchronize()
        means.append(e0.elapsed_time(e1) / reps)
    return means


def run_ladder(args):
    """The pages' benchmark table ("LeetGPU problem 2: matrix multiplication",
    yekq.top, section "benchmark summary": each version warmed up once, then
    the mean of 10 runs, GFLOPS = 2MNK/t, % of cuBLAS) re-measured on this
    GPU: the pages' kernels v0..v4 (gemm_f32_ladder), this library's three
    modes (gemm_f32_ex) and, as context, torch.matmul (cuBLAS) in fp32 and
    with TF32 allowed.  Reported: the mean over batches of `--steps` calls
    (at least 10, the pages' count) and the median of the batch means."""
    import torch

    import accelerator_row_major_gb300 as g

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    rows = []
    for cfg in ("1024x512x1024", "1001x513x777"):
        p = workloads.PROBLEMS[cfg]
        A_h, B_h = workloads.problem_inputs(cfg)
        A = torch.from_numpy(A_h).to(dev)
        B = torch.from_numpy(B_h).to(dev)
        C = torch.empty((p.M, p.N), dtype=torch.float32, device=dev)
        flop = workloads.gemm_flops(p.M, p.N, p.K)
        cands = []
        for step in g.LADDER_STEPS:
            cands.append(("v%d" % step, "ladder_v%d" % step,
                          lambda step=step: g.check(g.gemm_f32_ladder(A, B, C, p.M, p.N, p.K, step, stream))))
        for mode in ("ffma", "tc3x", "tc1x"):
            cands.append((mode, None,
                          lambda mode=mode: g.check(g.gemm_f32_ex(A, B, C, p.M, p.N, p.K, mode, 0, stream))))

        def torch_mm(tf32):
            def fn():
                torch.backends.cuda.matmul.allow_tf32 = tf32
                torch.matmul(A, B, out=C)
            return fn
        cands.append(("torch.matmul fp32", "cuBLAS (context)", torch_mm(False)))
        cands.append(("torch.matmul tf32", "cuBLAS (context)", torch_mm(True)))
        results = []
        for name, kernel, fn in cands:
            times = time_calls(fn, stream, max(args.warmup, 3), max(args.steps, 10))   # batch means
            if kernel is None:
                kernel = g.gemm_f32_last_kernel()
            mean = statistics.fmean(times)
            results.append((name, kernel, mean, statistics.median(times)))
        torch.backends.cuda.matmul.allow_tf32 = False
        ref = next(r for r in results if r[0] == "torch.matmul fp32")[2]
        for name, kernel, mean, med in results:
            row = {"config": cfg, "shape": [p.M, p.K, p.N], "version": name, "kernel": kernel,
                   "mean_ms": round(mean, 5), "median_ms": round(med, 5),
                   "gflops_mean": round(flop / mean / 1e6, 1), "gflops_median": round(flop / med / 1e6, 1),
                   "pct_of_cublas_fp32": round(100.0 * ref / mean, 1),
                   "stat": "warm L2; %d warm-up calls, then 5 batches of %d calls, each batch timed "
                           "with CUDA events" % (max(args.warmup, 3), max(args.steps, 10))}
            rows.append(row)
            print(json.dumps(row), flush=True)
    sys.stderr.write("\n| size | version | kernel | mean ms | GFLOPS | % of torch fp32 |\n|---|---|---|---|---|---|\n")
    for r in rows:
        sys.stderr.write("| %s | %s | %s | %.4f | %.0f | %.1f |\n" % (
            "x".join(str(v) for v in r["shape"]), r["version"], r["kernel"], r["mean_ms"],
            r["gflops_mean"], r["pct_of_cublas_fp32"]))
    return 0


def run_sweep(args):
    """Every problem in every mode, as the measurement plan asks: warm L2
    (the same inputs back to back, as on the pages) and cold L2 (a buffer
    twice the L2 size written between calls), each call timed with CUDA
    events on the launching stream after 3 warm-up calls; mean and median
    over at least 20 calls, and the pages' own statistic (one warm-up, then
    the mean of 10 calls; "LeetGPU problem 2", section "test environment and timing")."""
    import torch

    import accelerator_row_major_gb300 as g

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(args.steps, 20)
    rows = []
    for cfg in ("100x37x70", "1024x512x1024", "1001x513x777", "4096x4096x4096", "8192x8192x8192",
                "65536x1024x64", "64x4096x65536"):
        p = workloads.PROBLEMS[cfg]
        A_h, B_h = workloads.problem_inputs(cfg)
        A = torch.from_numpy(A_h).to(dev)
        B = torch.from_numpy(B_h).to(dev)
        C = torch.empty((p.M, p.N), dtype=torch.float32, device=dev)
        flop = workloads.gemm_flops(p.M, p.N, p.K)
        for mode in ("tc3x", "ffma", "tc1x"):
            def call():
                g.check(g.gemm_f32_ex(A, B, C, p.M, p.N, p.K, mode, 0, stream))
            n = reps if flop < 1e12 or mode != "ffma" else max(3, reps // 10)

            def timed(count, flush):
                out = []
                for _ in range(count):
                    with torch.cuda.stream(stream):
                        if flush:
                            scratch.zero_()
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        call()
                        e1.record(stream)
                    e1.synchronize()
                    out.append(e0.elapsed_time(e1))
                return out
            timed(3, False)
            warm = timed(n, False)
            cold = timed(n, True)
            timed(1, False)
            pages = statistics.fmean(timed(10, False))
            kernel = g.gemm_f32_last_kernel()
            row = {"config": cfg, "shape": [p.M, p.K, p.N], "mode": mode, "kernel": kernel,
                   "warm_mean_ms": round(statistics.fmean(warm), 5),
                   "warm_median_ms": round(statistics.median(warm), 5),
                   "cold_mean_ms": round(statistics.fmean(cold), 5),
                   "cold_median_ms": round(statistics.median(cold), 5),
                   "pages_stat_ms": round(pages, 5), "calls": n,
                   "tflops_warm_median": round(flop / statistics.median(warm) / 1e9, 2),
                   "tflops_cold_median": round(flop / statistics.median(cold) / 1e9, 2)}
            rows.append(row)
            print(json.dumps(row), flush=True)
        del A, B, C
        torch.cuda.empty_cache()
    sys.stderr.write("\n| problem | mode | kernel | warm median ms | cold median ms | pages' stat ms | TFLOPS warm / cold |\n"
                     "|---|---|---|---|---|---|---|\n")
    for r in rows:
        sys.stderr.write("| %s | %s | %s | %.4f | %.4f | %.4f | %.1f / %.1f |\n" % (
            r["config"], r["mode"], r["kernel"],
            r["warm_median_ms"], r["cold_median_ms"], r["pages_stat_ms"],
            r["tflops_warm_median"], r["tflops_cold_median"]))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_table:
        return run_oracle_table(args)
    if args.sweep:
        return run_sweep(args)
    if args.ladder:
        return run_ladder(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
