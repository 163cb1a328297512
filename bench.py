"""Benchmark: FP32 matrix multiply throughput (TFLOP/s = 2MNK / time) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]
    python bench.py --sweep [--sweep-workloads NAME ...]   # ablation table, one JSON line per run
    python bench.py --cpu-table [--cpu-seconds S]          # the oracle on every named problem
    python bench.py --e2e-only [--workload NAME]           # the host-buffer leg alone (profiling)
    python bench.py --kernel-only [--workload NAME]        # the device leg alone (profiling)

One step is one C = A x B call on the named workload (default: the square
4096^3 problem with standard-normal inputs, seed 3).  Inputs are resident in
HBM before timing.  Between timed steps L2 is flushed by writing a 512 MiB
buffer; each step is bracketed by CUDA events on the launching stream and the
flush lies outside the bracket.  Rank 0 prints one JSON line; after the timed
region it also times every other named problem the same way (``per_config``).

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica on its own GPU (the product does not shard across GPUs); the timed
region is bracketed by a barrier and synchronisation, and the slowest rank's
time counts.

``--impl reference`` times the CPU oracle (the double-accumulating triple
loop) on a bounded sample of rows of the same workload, on the host cores.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import PROBLEMS, problem_operands  # noqa: E402

METRIC = "SGEMM TFLOPS (2MNK/s) and % of FP32 roofline at 1024^3-8192^3 on 1 GB300"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "square_4096"
L2_FLUSH_BYTES = 512 << 20
# FP32 CUDA-core roofline derived from unit counts and clock: 152 SMs x 128 FP32
# lanes x 2 flops per FMA x 2070 MHz (maximum SM clock).
SMS, FP32_LANES_PER_SM, SM_MAX_MHZ = 152, 128, 2070.0
DERIVED_FP32_PEAK_TFLOPS = SMS * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
KERNEL_SOURCES = ["sgemm_ffma.cuh", "ptx.cuh", "res_maps.cuh", "sgemm_ffma_tma.cu", "sgemm_ffma_scaled.cu", "sgemm_ffma_tma_x.cu"]
# Nominal dense TF32 tensor rate of GB300 (context for the three-product entry).
TF32_DENSE_NOMINAL_TFLOPS = 1100.0


# ----------------------------------------------------------------- distributed helpers

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank float over the process group (identity without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------- clocks sampler

class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.cmd = ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", str(period_ms)]
        self.proc = None
        self.lines: list[str] = []
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        for t, line in self.lines:
            if self.t0 is not None and not (self.t0 <= t <= (self.t1 or t) + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- oracle (CPU) timing

def oracle_rows_rate(A, B, rows, threads):
    """Times the oracle on whole rows with `threads` host threads; returns
    (seconds, flops)."""
    import oracle

    t = time.perf_counter()
    oracle.default().gemm_rows_f64(A, B, rows, threads=threads)
    dt = time.perf_counter() - t
    return dt, 2.0 * len(rows) * B.shape[1] * A.shape[1]


def cpu_baseline(p, target_s: float = 12.0, threads: int | None = None):
    """The oracle, as it stands, on a bounded sample of output rows (all host
    cores unless `threads` is given)."""
    import numpy as np

    import oracle

    A, B = problem_operands(p)
    A, B = A.numpy(), B.numpy()
    threads = threads or oracle.default_threads()
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(p.M, size=min(p.M, max(threads, 8)), replace=False))
    dt, _ = oracle_rows_rate(A, B, probe, threads)
    per_row = dt / len(probe)
    n = int(min(p.M, max(len(probe), target_s / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(p.M, size=n, replace=False))
    dt, flops = oracle_rows_rate(A, B, rows, threads)
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {p.M} output rows of the {p.M}x{p.N}x{p.K} product "
                      f"(double accumulation, {dt:.1f} s)"}


# ----------------------------------------------------------------- traffic record

def _code_only(text: str) -> str:
    """C++ source without comments and whitespace (string literals in these
    files hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_source_digest() -> str:
    """Digest of the code (not the comments) of the product kernel's sources:
    a recorded DRAM-traffic figure applies while this digest is unchanged."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "dense_fp32_gemm_f32_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, variant: str):
    """DRAM bytes per launch from the committed ncu record, if it matches the
    current kernel source, workload and variant; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    for r in rec.get("records", []):
        if (r.get("workload") == workload and r.get("variant") == variant
                and r.get("kernel_src") == kernel_source_digest()):
            return r.get("dram_bytes_per_launch")
    return None


# ----------------------------------------------------------------- the two arms

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np

    import oracle

    p = PROBLEMS[args.workload]
    A, B = problem_operands(p)
    A, B = A.numpy(), B.numpy()
    threads = oracle.default_threads()
    rng = np.random.default_rng(1)
    # size each step so that warmup + steps take about two minutes in total
    probe = np.sort(rng.choice(p.M, size=min(p.M, max(threads, 8)), replace=False))
    dt, _ = oracle_rows_rate(A, B, probe, threads)
    per_row = dt / len(probe)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n = int(min(p.M, max(threads, budget / max(per_row, 1e-9))))
    times, flops = [], 0.0
    for i in range(args.warmup + args.steps):
        rows = np.sort(rng.choice(p.M, size=n, replace=False))
        t, f = oracle_rows_rate(A, B, rows, threads)
        if i >= args.warmup:
            times.append(t)
            flops = f
    ms = 1e3 * statistics.mean(times)
    value = flops / (ms / 1e3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(p, l2="n/a (host)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} of {p.M} output rows per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def pct(xs, q):
    """q-th percentile (nearest rank) of a list of numbers."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q / 100 * (len(ys) - 1)))))]


def run_e2e_only(args):
    """The end-to-end leg alone (sgemm_f32_host on pinned host buffers of the
    named workload, --warmup untimed then --steps timed calls), for profiling
    its pipeline of copies and products; prints one diagnostic JSON line."""
    import torch

    import dense_fp32_gemm_f32_gb300 as g

    torch.cuda.set_device(0)
    p = PROBLEMS[args.workload]
    A_cpu, B_cpu = problem_operands(p)
    A_pin, B_pin = A_cpu.pin_memory(), B_cpu.pin_memory()
    C_pin = torch.empty((p.M, p.N), dtype=torch.float32, pin_memory=True)
    for _ in range(args.warmup):
        g.sgemm_f32_host(A_pin, B_pin, C_pin)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        g.sgemm_f32_host(A_pin, B_pin, C_pin)
    dt = (time.perf_counter() - t0) / args.steps
    print(json.dumps({"leg": "e2e", "workload": p.name, "ms_per_step": 1e3 * dt,
                      "tflops": p.flops / dt / 1e12, "steps": args.steps, "warmup": args.warmup}), flush=True)
    return 0


def run_kernel_only(args):
    """The device leg alone (sgemm_f32 on the named workload's inputs resident
    in HBM, --warmup untimed then --steps timed calls, L2 flushed before
    each), for profiling one configuration's kernel; prints one diagnostic
    JSON line."""
    import torch

    import dense_fp32_gemm_f32_gb300 as g

    torch.cuda.set_device(0)
    p = PROBLEMS[args.workload]
    A_cpu, B_cpu = problem_operands(p)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    C = torch.empty((p.M, p.N), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    for i in range(args.warmup):
        flush.fill_(float(i))
        g.sgemm_f32(A, B, C)
    torch.cuda.synchronize()
    ms = []
    for i in range(args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.sgemm_f32(A, B, C)
        e1.record()
        ms.append((e0, e1))
    torch.cuda.synchronize()
    assert g.check_status() == 0
    t = statistics.median(a.elapsed_time(b) for a, b in ms)
    print(json.dumps({"leg": "kernel", "workload": p.name, "variant": g.describe(A, B, C), "ms_median": t,
                      "tflops": p.flops / (t / 1e3) / 1e12, "steps": args.steps, "warmup": args.warmup}),
          flush=True)
    return 0


def run_cpu_table(args):
    """The oracle timed on every named problem, on all host cores and on one
    core, each on a bounded sample of output rows (a few seconds); one JSON
    line per problem and core count.  Host only: no GPU is used."""
    import oracle

    for name, p in PROBLEMS.items():
        if name.endswith("_int"):
            continue
        for threads in (oracle.default_threads(), 1):
            rec = cpu_baseline(p, target_s=args.cpu_seconds, threads=threads)
            rec.update({"workload": name, "flops": p.flops})
            print(json.dumps(rec), flush=True)
    return 0


def per_config_records(lib, _lib, device, stream, flush, fma_peak, target_ms: float = 800.0):
    """Every named problem (not the integer twins) through sgemm_f32 and
    sgemm_3xtf32 on the C ABI: inputs resident in HBM, L2 flushed before each
    call (outside the event bracket), CUDA events on the launching stream.
    The number of timed calls per problem is sized so that each problem's
    timed calls take about ``target_ms`` (10 to 200 calls)."""
    import torch

    import dense_fp32_gemm_f32_gb300 as g

    sp = stream.cuda_stream
    out = {}
    for name, p in PROBLEMS.items():
        if name.endswith("_int"):
            continue
        A_cpu, B_cpu = problem_operands(p)
        A, B = A_cpu.to(device), B_cpu.to(device)
        C = torch.empty((p.M, p.N), dtype=torch.float32, device=device)
        rec = {"M": p.M, "N": p.N, "K": p.K, "dist": p.dist, "seed": p.seed, "variant": g.describe(A, B, C)}
        for entry in ("sgemm_f32", "sgemm_3xtf32"):
            fn = getattr(lib, entry)

            def call():
                _lib.check(fn(p.M, p.N, p.K, A.data_ptr(), p.K, B.data_ptr(), p.N, C.data_ptr(), p.N, sp), entry)

            for _ in range(3):
                call()
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            steps = int(min(200, max(10, target_ms / max(e0.elapsed_time(e1), 1e-3))))
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            for i in range(steps):
                flush.fill_(float(i))
                starts[i].record(stream)
                call()
                ends[i].record(stream)
            torch.cuda.synchronize(device)
            assert g.check_status() == 0, f"{name} {entry}: kernel status"
            ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
            tf = p.flops / (statistics.mean(ms) / 1e3) / 1e12
            if entry == "sgemm_f32":
                rec.update({"tflops": tf, "frac": tf / fma_peak, "frac_of_derived": tf / DERIVED_FP32_PEAK_TFLOPS,
                            "ms": {"mean": statistics.mean(ms), "median": statistics.median(ms),
                                   "p10": pct(ms, 10), "p90": pct(ms, 90)}, "steps": steps})
            else:
                rec["sgemm_3xtf32_tflops"] = tf
        out[name] = rec
        del A, B, C
    return out


def host_link_rates(device, stream, nbytes: int = 256 << 20, reps: int = 5):
    """Host<->device copy rate of one large pinned copy per direction (one
    cudaMemcpyAsync each, CUDA events, best of ``reps``), GB/s."""
    import torch

    h = torch.empty(nbytes // 4, dtype=torch.float32, pin_memory=True)
    d = torch.empty(nbytes // 4, dtype=torch.float32, device=device)
    rates = {}
    for name, dst, src in (("h2d_gbs", d, h), ("d2h_gbs", h, d)):
        best = None
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        rates[name] = nbytes / (best / 1e3) / 1e9
    rates["bytes_per_copy"] = nbytes
    return rates


def workload_config(p, l2):
    return {"workload": f"{p.name}: C = A x B, M={p.M} N={p.N} K={p.K}, row-major float32, "
                        f"A,B {p.dist} seed {p.seed}, C overwritten",
            "M": p.M, "N": p.N, "K": p.K, "dist": p.dist, "seed": p.seed, "l2": l2}


def run_ours(args, rank, world, local_rank):
    import torch

    import dense_fp32_gemm_f32_gb300 as g
    from dense_fp32_gemm_f32_gb300 import _lib

    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    lib = _lib.load()
    p = PROBLEMS[args.workload]
    A_cpu, B_cpu = problem_operands(p)
    A = A_cpu.to(device)
    B = B_cpu.to(device)
    C = torch.empty((p.M, p.N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream
    variant = g.describe(A, B, C)

    # FP32 FMA peak microbenchmark (both instruction forms), for context.
    import ctypes

    scratch = torch.empty(SMS * 8 * 256, dtype=torch.float32, device=device)
    peaks = {}
    for paired in (0, 1):
        fl = ctypes.c_double(0)
        for _ in range(2):
            _lib.check(lib.sgemm_bench_fma_peak(paired, SMS * 8, 4096, scratch.data_ptr(), sp, ctypes.byref(fl)),
                       "fma peak")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        reps = 5
        for _ in range(reps):
            lib.sgemm_bench_fma_peak(paired, SMS * 8, 4096, scratch.data_ptr(), sp, ctypes.byref(fl))
        e1.record(stream)
        e1.synchronize()
        peaks["ffma2" if paired else "ffma"] = fl.value * reps / (e0.elapsed_time(e1) / 1e3) / 1e12

    def step():
        _lib.check(lib.sgemm_f32(p.M, p.N, p.K, A.data_ptr(), p.K, B.data_ptr(), p.N, C.data_ptr(), p.N, sp),
                   "sgemm_f32")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert g.check_status() == 0

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        barrier(device)
        torch.cuda.synchronize()
        clk.mark_start()
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(float(i))  # write > L2 so every step starts cold
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier(device)
        wall = time.perf_counter() - t_wall
        clk.mark_end()
    status = g.check_status()
    assert status == 0, f"kernel status {status}"
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_local = statistics.mean(kernel_ms)
    ms = max_over_ranks(ms_local, device)
    value = world * p.flops / (ms / 1e3) / 1e12
    # Kernels one sgemm_f32 call launches (the memset of the stream-K flags
    # is not a kernel): the product, plus A's transposing copy ("/at") and the
    # repacking copy ("/repack") when the plan has them.
    kernels_per_call = 1 + ("/at" in variant) + ("/repack" in variant)

    # The dominant kernel alone.  With "/at" the call first copies A
    # transposed; the product kernel is then timed by itself by giving it an
    # A already stored transposed (sgemm_f32_gemm with transa: the same kernel,
    # plan and launch, without the copy), over the same number of steps and
    # with the same L2 flush.
    if "/at" in variant:
        At = A.t().contiguous()

        def step_kernel():
            _lib.check(lib.sgemm_f32_gemm(1, 0, p.M, p.N, p.K, 1.0, At.data_ptr(), p.M, B.data_ptr(), p.N, 0.0,
                                          C.data_ptr(), p.N, sp), "sgemm_f32_gemm")

        for _ in range(3):
            step_kernel()
        k_starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        k_ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(float(i))
            k_starts[i].record(stream)
            step_kernel()
            k_ends[i].record(stream)
        torch.cuda.synchronize()
        assert g.check_status() == 0
        product_ms = [s_.elapsed_time(e_) for s_, e_ in zip(k_starts, k_ends)]
        del At
        kernel_timing = ("product kernel alone: the same launch on an A stored transposed "
                         "(sgemm_f32_gemm transa), CUDA events, same steps and L2 flush")
    else:
        product_ms = kernel_ms
        kernel_timing = "the whole call (one kernel launch per step), CUDA events"
    achieved = p.flops / (statistics.mean(product_ms) / 1e3) / 1e12

    # The tensor-core entry on the same workload, timed the same way (reported
    # beside the main line, not as it: the FP32 FFMA kernel is the headline).
    def step_tc():
        _lib.check(lib.sgemm_3xtf32(p.M, p.N, p.K, A.data_ptr(), p.K, B.data_ptr(), p.N, C.data_ptr(), p.N, sp),
                   "sgemm_3xtf32")

    for _ in range(3):
        step_tc()
    tc_ms = []
    for i in range(max(3, min(args.steps, 50))):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_tc()
        e1.record(stream)
        e1.synchronize()
        tc_ms.append(e0.elapsed_time(e1))
    assert g.check_status() == 0
    tc_tflops = p.flops / (statistics.mean(tc_ms) / 1e3) / 1e12

    # End to end through the host-buffer entry: pinned host A, B -> device,
    # multiply, C -> pinned host, every step.
    A_pin, B_pin = A_cpu.pin_memory(), B_cpu.pin_memory()
    C_pin = torch.empty((p.M, p.N), dtype=torch.float32, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        g.sgemm_f32_host(A_pin, B_pin, C_pin, device=device)
    barrier(device)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        g.sgemm_f32_host(A_pin, B_pin, C_pin, device=device)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, device)
    e2e_value = world * p.flops / e2e_s / 1e12
    link = host_link_rates(device, stream)

    # Every named problem, timed the same way (after the headline's timed
    # region; rank 0 only).
    fma_peak = max(peaks.values())
    per_config = per_config_records(lib, _lib, device, stream, flush, fma_peak) if rank == 0 else None

    if rank != 0:
        return 0
    cpu = cpu_baseline(p) if world == 1 else None
    clocks = clk.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(p, l2=f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write)"),
        "variant": variant,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": fma_peak, "unit": UNIT,
                     "frac": achieved / fma_peak,
                     "traffic": recorded_traffic(p.name, variant),
                     "peak_source": "measured in this run: the larger of the FFMA and paired-FFMA "
                                    "microbenchmarks (all SMs, 8 warps each, independent FMA chains)",
                     "measured_fma_peak": peaks,
                     "peak_derived": DERIVED_FP32_PEAK_TFLOPS,
                     "frac_of_derived": achieved / DERIVED_FP32_PEAK_TFLOPS,
                     "peak_derived_source": "152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz",
                     "algorithmic_flops_per_launch": p.flops, "min_bytes_per_launch": p.min_bytes,
                     "kernel_ms": statistics.mean(product_ms), "kernel_timing": kernel_timing},
        "secondary": {"sgemm_3xtf32": {
            "value": tc_tflops, "unit": UNIT, "ms": statistics.mean(tc_ms),
            "note": "three TF32 tensor-core products per FP32 product; same accuracy contract",
            "frac_of_tf32_dense_nominal_over_3": tc_tflops / (TF32_DENSE_NOMINAL_TFLOPS / 3)}},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": 4 * (p.M * p.K + p.K * p.N),
                "d2h_bytes_per_step": 4 * p.M * p.N, "ms_per_step": 1e3 * e2e_s,
                "timing": "host wall clock over the steps, each ending in a stream synchronisation",
                "link": link},
        "gpu_launches": args.steps * kernels_per_call,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "wall_s_timed_region": wall,
        "kernel_ms": {"mean": ms_local, "min": min(kernel_ms), "p10": pct(kernel_ms, 10),
                      "median": statistics.median(kernel_ms), "p90": pct(kernel_ms, 90), "max": max(kernel_ms)},
    }
    print(json.dumps(line), flush=True)
    return 0


# sgemm_3xtf32 kernels: 1 = split-tile (also with its K split off), 2 = direct-A, 3 = split-tile on 128 x 256
# tiles, 4 = 3 with B pre-split.
SWEEP_TF32X3 = [{"variant": 1, "split_k": 1}, {"variant": 1}, {"variant": 2}, {"variant": 3}, {"variant": 4}]
SWEEP_OPTIONS = [
    {},
    {"producer": 1},
    {"math": 1},
    {"stages": 1},
    {"stages": 2},
    {"stages": 6},
    {"producer": 2},
    {"producer": 3},
    {"producer": 3, "split_k": 1},
    {"tile_n": 256},
    {"tile_n": 256, "stages": 2},
    {"tile_n": 256, "stages": 3},
    {"tile_n": 256, "split_k": 1},
    {"tile_n": 64},
    {"tile_n": 64, "stages": 3},
    {"tile_n": 64, "stages": 2},
    {"tile_n": 64, "split_k": 1},
    {"repack": 1},
    {"repack": 2},
    {"producer": 7},
    {"a_layout": 1},
    {"a_layout": 2, "tile_n": 256},
    {"producer": 5},
    {"producer": 5, "stages": 3},
    {"producer": 6},
    {"split_k": 1},
    {"split_k": 2},
    {"split_k": 4},
    {"split_k": 8},
    {"tail_split": 4},
    {"stream_k": 2},
    {"tile_k": 16},
    {"tile_k": 16, "stages": 2},
    {"tile_k": 16, "stages": 6},
    {"group_m": 1},
    {"l2_hint": 1},
    {"l2_hint": 2},
    {"producer": 8},
    {"edge": 1},
]


def run_sweep(args):
    """Ablations: every named workload x the forced variants of sgemm_f32_ex.
    Median of ``--steps`` event-timed launches, L2 flushed before each."""
    import torch

    import dense_fp32_gemm_f32_gb300 as g

    torch.cuda.set_device(0)
    torch.backends.cuda.matmul.allow_tf32 = False  # the library comparison runs in full FP32
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    names = args.sweep_workloads or [n for n in PROBLEMS if not n.endswith("_int")]
    # An idle GPU runs the first calls below its working clock: keep it busy
    # for a second before the first measurement.
    t_end = time.perf_counter() + 1.0
    while time.perf_counter() < t_end:
        flush.fill_(0.0)
        torch.cuda.synchronize()
    for name in names:
        p = PROBLEMS[name]
        A_cpu, B_cpu = problem_operands(p)
        A, B = A_cpu.cuda(), B_cpu.cuda()
        C = torch.empty((p.M, p.N), dtype=torch.float32, device="cuda")
        runs = [(opt, (lambda o=opt: g.sgemm_f32_ex(A, B, C, **o)) if opt else (lambda: g.sgemm_f32(A, B, C)))
                for opt in SWEEP_OPTIONS]
        runs += [({"entry": "sgemm_3xtf32", **o}, lambda o=o: g.sgemm_3xtf32_ex(A, B, C, **o)) for o in SWEEP_TF32X3]
        # The general entry: alpha = 1.5, beta = 0.5 (C read and written) in
        # each storage order (a transposed operand is copied transposed first).
        At, Bt = A.t().contiguous(), B.t().contiguous()
        runs += [({"entry": "sgemm_f32_gemm", "transa": ta, "transb": tb, "alpha": 1.5, "beta": 0.5},
                  lambda ta=ta, tb=tb: g.sgemm_f32_gemm(At if ta else A, Bt if tb else B, C, alpha=1.5, beta=0.5,
                                                        transa=ta, transb=tb))
                 for ta, tb in ((0, 0), (1, 0), (0, 1), (1, 1))]
        # Context only (a library GEMM, on no path of this project): the
        # FP32 GEMM torch runs with TF32 disabled, timed the same way.
        runs += [({"entry": "torch.mm", "tf32": False}, lambda: torch.mm(A, B, out=C))]
        # Sizes whose working set fits in L2: the automatic choice also with
        # the operands left warm in L2 (no flush between calls).
        warm = p.flops <= 2 * 2048**3
        for opt, run in runs:
            try:
                for _ in range(3):
                    run()
                torch.cuda.synchronize()
                ts = []
                for i in range(args.steps):
                    flush.fill_(float(i))
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    run()
                    e1.record()
                    e1.synchronize()
                    ts.append(e0.elapsed_time(e1))
                assert g.check_status() == 0
                ms = statistics.median(ts)
                tf = p.flops / (ms / 1e3) / 1e12
                rec = {"workload": name, "options": opt, "ms": ms, "tflops": tf,
                       "frac_of_derived_peak": tf / DERIVED_FP32_PEAK_TFLOPS}
            except Exception as e:  # an option the shape does not allow
                rec = {"workload": name, "options": opt, "error": str(e)}
            print(json.dumps(rec), flush=True)
        if warm:
            # Back to back without flushing (operands warm in L2), timed as one
            # batch of --steps calls, so that no host launch gap is counted.
            for opt, run in ((dict(l2="warm"), lambda: g.sgemm_f32(A, B, C)),
                             (dict(entry="torch.mm", tf32=False, l2="warm"), lambda: torch.mm(A, B, out=C))):
                for _ in range(3):
                    run()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    run()
                e1.record()
                e1.synchronize()
                assert g.check_status() == 0
                ms = e0.elapsed_time(e1) / args.steps
                tf = p.flops / (ms / 1e3) / 1e12
                print(json.dumps({"workload": name, "options": opt, "ms": ms, "tflops": tf,
                                  "frac_of_derived_peak": tf / DERIVED_FP32_PEAK_TFLOPS}), flush=True)
        del A, B, C, At, Bt
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(PROBLEMS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--sweep", action="store_true", help="print the ablation table instead")
    ap.add_argument("--sweep-workloads", nargs="*", choices=sorted(PROBLEMS), default=None)
    ap.add_argument("--cpu-table", action="store_true",
                    help="time the oracle on every named problem, all cores and one core (host only)")
    ap.add_argument("--cpu-seconds", type=float, default=4.0, help="bounded sample per --cpu-table entry")
    ap.add_argument("--e2e-only", action="store_true",
                    help="time only the end-to-end leg (host buffers) of --workload; a diagnostic line")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the device leg (sgemm_f32 on resident inputs) of --workload; a diagnostic line")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if args.sweep:
        return run_sweep(args)
    if args.e2e_only:
        return run_e2e_only(args)
    if args.kernel_only:
        return run_kernel_only(args)
    if args.cpu_table:
        return run_cpu_table(args)
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch

            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_ours(args, rank, world, local_rank)
    finally:
        import torch.distributed as dist

        if dist.is_available() and dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
