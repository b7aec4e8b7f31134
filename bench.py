#!/usr/bin/env python3
"""Benchmark of the FP32 SGEMM on GB300: one JSON line on stdout (rank 0).

A step is one sgemm() call (A-transpose pre-pass + main kernel) on the timed
workload: M = N = K = 8192, row-major fp32, A, B, C_in ~ U[-1, 1) from seed
1003, alpha = 1.5, beta = 0.5.  Inputs (805 MB) are larger than the 129 MB L2,
so no flush is needed between steps.

  value    GFLOP/s = 2MNK / (device time per step), inputs resident in HBM,
           summed over ranks (replicas: every rank runs the whole workload)
  e2e      the same metric through the host-buffer entry point sgemm_host():
           pinned host A, B, C_in copied in and C copied out every step
  roofline the main kernel against the FP32 FFMA peak (SMs x 128 FFMA/clk x
           2 FLOP x 2070 MHz), timed with CUDA events on its own stream
  cpu_baseline  the CPU oracle on this host's cores on a bounded sample of rows

`--impl reference` times the CPU oracle (the only reference implementation) on
a bounded sample of the same workload per step and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
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

METRIC = "SGEMM GFLOP/s (2MNK/t) at M=N=K=8192 FP32; % of GB300 FP32 FFMA peak"
FFMA_PER_SM_PER_CLK = 128
SM_MAX_MHZ_FALLBACK = 2070.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "traffic.json")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
# nominal dense TF32 / BF16 tensor throughput of GB300 (1.1 / 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25
# The TF32 MMA rate of one SM as a stand-alone probe measured it on GB300: one
# tcgen05.mma kind::tf32 of M 128, N 256, K 8 every 128 cycles = 2048 MAC =
# 4096 FLOP per clock per SM (profiles/sgemm_3xtf32_8192.md).
TF32_MMA_FLOP_PER_SM_PER_CLK = 4096
BF16_FALLBACK_TFLOPS = 1900.0
HBM_FALLBACK_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, help="workload name (default: the 8192^3 case)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-tf32x3", action="store_true",
                    help="skip the 3xTF32 tensor-core measurement added to the default line")
    ap.add_argument("--path", choices=["ffma", "tf32x3"], default="ffma",
                    help="ffma: the FP32 FFMA kernel (the headline); tf32x3: the 3xTF32 "
                         "tensor-core entry point, same tolerance, its own roofline")
    ap.add_argument("--variant", type=int, default=-1,
                    help="force a kernel variant (tile-configuration sweeps); -1 = automatic")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle on every workload with all host cores and with "
                         "one, print one JSON line and exit (no GPU work)")
    ap.add_argument("--oracle-budget", type=float, default=2.0,
                    help="seconds of oracle work per --oracle-table measurement")
    return ap.parse_args()


# ---------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(world, value, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gflops(flops_per_step, ms_per_step_max, world):
    """Whole-job rate: every rank runs the full workload (replicas), the step
    time is the slowest rank's, so the job does world x flops per step."""
    return flops_per_step / (ms_per_step_max * 1e-3) / 1e9 * world


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 100 ms; only samples inside [t0, t1] are kept."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.windows = []

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, windows=None):
        """Clock summary over the samples inside `windows` (default: every
        marked window); the sample file is read once and kept."""
        import datetime
        if not hasattr(self, "_rows"):
            self._rows = []
            if self.path and os.path.exists(self.path):
                for line in open(self.path):
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        self._rows.append((ts, float(parts[2]), float(parts[3]), parts[4], parts[5:]))
                    except ValueError:
                        continue
                os.unlink(self.path)
        rows = self._rows
        windows = self.windows if windows is None else windows
        inside = [r for r in rows if any(t0 - 0.15 <= r[0] <= t1 + 0.15 for t0, t1 in windows)]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for n, v in zip(names, r[4][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        power = []
        for r in use:
            try:
                power.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use),
                "in_window": bool(inside),
                "power_w_median": statistics.median(power) if power else None}


# ---------------------------------------------------------------------- CPU oracle timing
def l2_note(w):
    """How the timed steps avoid a warm L2: the bytes of A, B and C per step."""
    lda, ldb, ldc = w.lds()
    mb = 4.0 * w.batch * (w.M * lda + w.K * ldb + w.M * ldc) / 1e6
    if mb > 129.0:
        return f"inputs larger than L2 (A, B, C {mb:.0f} MB vs 129 MB), no flush"
    return f"A, B, C {mb:.0f} MB, not larger than the 129 MB L2: no flush, L2 partly warm"


def time_e2e(step, w, steps, world, device, entry_point, h2d_bytes, d2h_bytes):
    """End-to-end timing of a host-buffer call: two untimed calls, then `steps`
    calls timed one by one on the host clock (each call returns with C on the
    host).  The value is taken at the median call (host-side copies make single
    calls noisy); the mean and the minimum are reported beside it."""
    for _ in range(2):
        step()
    barrier(world, device)
    times = []
    for _ in range(steps):
        t = time.perf_counter()
        step()
        times.append(time.perf_counter() - t)
    med = max_over_ranks(world, statistics.median(times), device)
    mean = max_over_ranks(world, sum(times) / len(times), device)
    return {"value": round(w.flops / med / 1e9 * world, 3), "unit": "GFLOP/s",
            "entry_point": entry_point, "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes, "ms_per_step": round(med * 1e3, 3),
            "ms_mean": round(mean * 1e3, 3), "ms_min": round(min(times) * 1e3, 3),
            "statistic": "median of the timed calls"}


def oracle_rows_fn(w, A, B, C, threads=None):
    """f(idx): the oracle as it stands on full rows idx of the workload (batch 0
    of a batched one, with its bias and activation); `threads` host threads
    (default: all)."""
    import oracle
    from dense_fp32_gemm_02_gb300.workloads import workload_bias
    if w.extended:
        bias = workload_bias(w)
        A0, B0 = (A[0], B[0]) if w.batch > 1 else (A, B)
        C0 = None if (C is None or w.beta == 0) else (C[0] if w.batch > 1 else C)
        b0 = None if bias is None else bias[0]
        return lambda idx: oracle.sgemm_ex_rows(A0, B0, C0, w.alpha, w.beta, b0, w.act, idx,
                                                threads=threads, with_bound=False)
    c_in = C if w.beta != 0 else None
    return lambda idx: oracle.sgemm_rows(A, B, c_in, w.alpha, w.beta, idx, threads=threads,
                                         with_bound=False)


def time_oracle_rows(w, A, B, C, row_budget_s=12.0, first=16, max_rows=None, threads=None):
    """The oracle as it stands on full rows of the workload; grows the sample
    until about `row_budget_s` seconds of CPU work.  Returns (gflops, rows, secs)."""
    import numpy as np
    rows_fn = oracle_rows_fn(w, A, B, C, threads)
    rows_done, secs, r0 = 0, 0.0, 0
    n = first
    max_rows = max_rows or w.M
    while rows_done < max_rows:
        n = min(n, max_rows - rows_done)
        idx = np.arange(r0, r0 + n, dtype=np.int64)
        t = time.perf_counter()
        rows_fn(idx)
        secs += time.perf_counter() - t
        rows_done += n
        r0 += n
        if secs >= row_budget_s:
            break
        n *= 2
    gflops = 2.0 * rows_done * w.N * w.K / secs / 1e9
    return gflops, rows_done, secs


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------- reference arm
def run_reference(args):
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    from dense_fp32_gemm_02_gb300.workloads import BENCH_WORKLOAD, WORKLOADS, workload_inputs
    w = WORKLOADS[args.workload or BENCH_WORKLOAD]
    A, B, C = workload_inputs(w)
    # enough full rows per step for every host core to get two
    rows_per_step = max(16, 2 * host_cores())
    rows_fn = oracle_rows_fn(w, A, B, C)

    def step(i):
        r0 = (i * rows_per_step) % w.M
        idx = np.arange(r0, min(r0 + rows_per_step, w.M), dtype=np.int64)
        rows_fn(idx)
        return len(idx)

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    rows = sum(step(args.warmup + i) for i in range(args.steps))
    secs = time.perf_counter() - t
    gflops = 2.0 * rows * w.N * w.K / secs / 1e9
    cores = host_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gflops, 3), "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64-accumulate", "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                   "beta": w.beta, "sample": f"{rows_per_step} full output rows per step"},
        "cpu_baseline": {"value": round(gflops, 3), "unit": "GFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{rows_per_step} rows x {w.N} cols x K={w.K} per step"},
        "e2e": {"value": round(gflops, 3), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- oracle table
def cpu_model():
    """The host CPU's model line from /proc/cpuinfo, or the platform's name."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def run_oracle_table(args):
    """The oracle as it stands, on every workload, once with all host cores and
    once with one: GFLOP/s on a bounded sample of full output rows, and the time
    the whole oracle of that workload would take at that rate."""
    import platform
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return 0
    from dense_fp32_gemm_02_gb300.workloads import WORKLOADS, workload_inputs
    cores = host_cores()
    table = []
    for name, w in WORKLOADS.items():
        A, B, C = workload_inputs(w)
        for threads in (cores, 1):
            g, rows, secs = time_oracle_rows(w, A, B, C, row_budget_s=args.oracle_budget,
                                             first=max(1, min(16, threads)), threads=threads)
            table.append({"workload": name, "threads": threads, "gflops": round(g, 3),
                          "rows": rows, "secs": round(secs, 3),
                          "full_oracle_s": round(w.flops / (g * 1e9), 1)})
        del A, B, C
    print(json.dumps({"oracle_table": table, "unit": "GFLOP/s", "kind": "oracle",
                      "host": {"machine": platform.machine(), "cpu": cpu_model(),
                               "cores": cores}}), flush=True)
    return 0


# ---------------------------------------------------------------------- our arm
def load_traffic(workload_name):
    try:
        with open(PROFILE_SUMMARY) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e and e.get("kernel_revision") == kernel_revision():
            return e.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


def kernel_revision():
    """Hash of the CUDA sources; a stored ncu traffic figure only counts for
    the kernel it was measured on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_gemm_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()[:16]


def tensor_peak_tf32():
    """(peak TFLOP/s of TF32 MMA, source text): the measured dense bf16 burst
    peak times the nominal TF32/BF16 ratio."""
    try:
        with open(PEAKS_FILE) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
        src = f"measured bf16 burst {bf16} TFLOP/s x nominal tf32/bf16 ratio 1.1/2.25"
    except (OSError, ValueError, KeyError):
        bf16 = BF16_FALLBACK_TFLOPS
        src = f"fallback bf16 {bf16} TFLOP/s x nominal tf32/bf16 ratio 1.1/2.25"
    return bf16 * TF32_PER_BF16, src


def probed_mma_fields(achieved_tflops, sms, sm_mhz=None):
    """The 3xTF32 main kernel against the MMA unit's probed per-clock rate: at
    the 2070 MHz maximum SM clock and, when known, at the clock measured during
    its timed region.  The derived `peak` (bf16 burst x nominal ratio) sits
    below the unit's rate, so `frac` there can read above 1; these cannot."""
    peak = sms * TF32_MMA_FLOP_PER_SM_PER_CLK * SM_MAX_MHZ_FALLBACK * 1e6 / 1e12
    out = {"probed_mma_peak": round(peak, 3),
           "probed_mma_source": f"{sms} SMs x {TF32_MMA_FLOP_PER_SM_PER_CLK} TF32 FLOP/clk "
                                f"(probed: one M128 N256 K8 MMA per 128 cycles) x 2070 MHz",
           "frac_of_probed_mma": round(achieved_tflops / peak, 4) if achieved_tflops else None,
           "frac_of_probed_mma_at_measured_clock": None}
    if achieved_tflops and sm_mhz:
        at = sms * TF32_MMA_FLOP_PER_SM_PER_CLK * sm_mhz * 1e6 / 1e12
        out["frac_of_probed_mma_at_measured_clock"] = round(achieved_tflops / at, 4)
    return out


def hbm_peak_gbs():
    """(peak GB/s, source text): the measured copy bandwidth of this machine's
    GB300s, else the fallback figure."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured: MEASURED_PEAKS.json hbm_gbs (copy)"
    except (OSError, ValueError, KeyError):
        return HBM_FALLBACK_GBS, "fallback: 6.8 TB/s"


def dram_use(traffic, ms):
    """{dram_gbs, dram_frac}: one launch's DRAM bytes (the ncu figure) over its
    CUDA-event duration, and that rate against the measured copy bandwidth;
    both None without a traffic figure for the current kernel."""
    if not traffic or not ms or ms <= 0:
        return {"dram_gbs": None, "dram_frac": None}
    gbs = traffic / (ms * 1e-3) / 1e9
    peak, _ = hbm_peak_gbs()
    return {"dram_gbs": round(gbs, 1), "dram_frac": round(gbs / peak, 4)}


def measure_tf32x3(args, w, binding, dA, dB, dC, C, stream, world, device):
    """The 3xTF32 tensor-core entry point on the same workload: device-time
    rate, the main kernel against the TF32 tensor roofline, and end to end
    (pinned host buffers copied in and C copied out every step)."""
    import numpy as np
    import torch
    C0 = torch.from_numpy(np.ascontiguousarray(C)).to(device) if C is not None else None

    def reset():
        if C0 is not None:
            dC.copy_(C0)

    def step():
        binding.sgemm_3xtf32_into(dA, dB, dC, w.alpha, w.beta, stream=stream)

    reset()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    binding.profile_collect()
    binding.profile_enable(True)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    start.record(stream)
    for _ in range(args.steps):
        step()
    stop.record(stream)
    stop.synchronize()
    binding.profile_enable(False)
    prof = binding.profile_collect()
    if binding.device_status(stream=stream) != 0:
        raise RuntimeError("device error word set during the 3xTF32 timed region")
    ms = max_over_ranks(world, start.elapsed_time(stop), device) / args.steps
    main_ms = prof["main_ms"] / args.steps   # every compute launch of a step
    # all pre-pass launches of a step (split of A and split+transpose of B)
    split_ms = prof["pack_ms"] / args.steps
    peak, src = tensor_peak_tf32()
    mma_tflops = 3.0 * w.flops / (main_ms * 1e-3) / 1e12
    out = {
        "value": round(aggregate_gflops(w.flops, ms, world), 3), "unit": "GFLOP/s",
        "ms_per_step": round(ms, 4), "entry_point": "sgemm_3xtf32",
        "roofline": {"bound": "tensor", "kernel": "sgemm_3xtf32 main kernel (CTA pair or single CTA, chosen per shape)",
                     "achieved": round(mma_tflops, 3), "peak": round(peak, 3), "unit": "TFLOP/s",
                     "frac": round(mma_tflops / peak, 4), "traffic": load_traffic(w.name + ":tf32x3"),
                     **dram_use(load_traffic(w.name + ":tf32x3"), main_ms),
                     "peak_source": src,
                     "algorithmic_flops_per_launch": 3.0 * w.flops,
                     "note": "three TF32 MMAs per fp32 product: achieved counts MMA FLOPs",
                     "main_kernel_ms": round(main_ms, 4), "split_kernels_ms": round(split_ms, 4)},
    }
    if not args.no_e2e:
        # through the host-buffer entry point of this path (pipelined copies)
        hA = torch.from_numpy(np.ascontiguousarray(dA.cpu().numpy())).pin_memory()
        hB = torch.from_numpy(np.ascontiguousarray(dB.cpu().numpy())).pin_memory()
        hC = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
        if C0 is not None:
            hC.copy_(C0.cpu())

        def e2e_step():
            binding.sgemm_host(hA, hB, hC, w.alpha, w.beta, stream=stream, tensor_cores=True)

        out["e2e"] = time_e2e(e2e_step, w, args.steps, world, device, "sgemm_host_3xtf32",
                              (hA.numel() + hB.numel() + (hC.numel() if w.beta != 0 else 0)) * 4,
                              hC.numel() * 4)
    return out


def run_ours(args):
    import numpy as np
    import torch

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")

    from dense_fp32_gemm_02_gb300 import binding
    from dense_fp32_gemm_02_gb300.workloads import (BENCH_WORKLOAD, WORKLOADS, workload_bias,
                                                    workload_inputs)
    w = WORKLOADS[args.workload or BENCH_WORKLOAD]
    binding.set_variant(args.variant)
    A, B, C = workload_inputs(w)
    bias = workload_bias(w)
    if w.extended and args.path != "ffma":
        raise SystemExit("batched and fused-epilogue workloads run on the FFMA path (sgemm_ex)")
    props = torch.cuda.get_device_properties(device)
    sms = props.multi_processor_count
    stream = torch.cuda.Stream(device)

    dA = torch.from_numpy(np.ascontiguousarray(A)).to(device)
    dB = torch.from_numpy(np.ascontiguousarray(B)).to(device)
    dC = torch.from_numpy(np.ascontiguousarray(C)).to(device) if C is not None else \
        torch.zeros(((w.batch,) if w.batch > 1 else ()) + (w.M, w.N), device=device)
    dbias = torch.from_numpy(bias).to(device) if bias is not None else None
    torch.cuda.synchronize()

    gemm = binding.sgemm_into if args.path == "ffma" else binding.sgemm_3xtf32_into

    def step():
        if w.extended:
            binding.sgemm_ex_into(dA, dB, dC, w.alpha, w.beta, bias=dbias, act=w.act,
                                  stream=stream)
        else:
            gemm(dA, dB, dC, w.alpha, w.beta, stream=stream)

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if binding.device_status(stream=stream) != 0:
        raise RuntimeError("device error word set during warm-up")

    # ---- timed region (device time, inputs resident)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    binding.profile_collect()
    binding.profile_enable(True)
    launches0 = binding.kernel_launch_count()
    barrier(world, device)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        step()
    stop.record(stream)
    stop.synchronize()
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world, device)
    launches = binding.kernel_launch_count() - launches0
    binding.profile_enable(False)
    prof = binding.profile_collect()
    clocks.mark(t0, t1)
    ms = start.elapsed_time(stop)
    ms = max_over_ranks(world, ms, device)
    if binding.device_status(stream=stream) != 0:
        raise RuntimeError("device error word set during the timed region")

    ms_per_step = ms / args.steps
    gflops = aggregate_gflops(w.flops, ms_per_step, world)
    # Per-call median and minimum, from a second pass of the same steps
    # without any profiling: an event after every call and none inside it
    # (every event recorded between two kernels costs the GPU about 2 us, and
    # the timed region above already carries the library's three per call).
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    marks[0].record(stream)
    for i in range(args.steps):
        step()
        marks[i + 1].record(stream)
    marks[-1].synchronize()
    per_call = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    per_call_median = statistics.median(per_call)
    per_call_min = min(per_call)
    # the main kernel these calls ran (the library's own record of its launch)
    kernel_text = binding.last_kernel()

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and not w.extended:
        hA = torch.from_numpy(np.ascontiguousarray(A)).pin_memory()
        hB = torch.from_numpy(np.ascontiguousarray(B)).pin_memory()
        hC0 = torch.from_numpy(np.ascontiguousarray(C)) if C is not None else None
        hC = torch.empty((w.M, w.N), dtype=torch.float32).pin_memory()
        if hC0 is not None:
            hC.copy_(hC0)
        te0 = time.time()
        e2e = time_e2e(lambda: binding.sgemm_host(hA, hB, hC, w.alpha, w.beta, stream=stream),
                       w, args.steps, world, device, "sgemm_host",
                       (hA.numel() + hB.numel() + (hC.numel() if w.beta != 0 else 0)) * 4,
                       hC.numel() * 4)
        clocks.mark(te0, time.time())
    main_windows = list(clocks.windows)
    tf32x3 = None
    if args.path == "ffma" and not args.no_tf32x3 and not w.extended:
        t0x = time.time()
        tf32x3 = measure_tf32x3(args, w, binding, dA, dB, dC, C, stream, world, device)
        tf_window = (t0x, time.time())
        clocks.mark(*tf_window)
    clocks.stop()
    clk = clocks.summary(main_windows)
    if tf32x3 is not None:
        tclk = clocks.summary([tf_window])
        tf32x3["clocks"] = {"sm_mhz": tclk.get("sm_mhz"), "sm_max_mhz": tclk.get("sm_max_mhz"),
                            "reasons": tclk.get("reasons"), "samples": tclk.get("samples"),
                            "power_w_median": tclk.get("power_w_median")}
        tf32x3["roofline"].update(probed_mma_fields(tf32x3["roofline"]["achieved"], sms,
                                                    tclk.get("sm_mhz")))

    # ---- roofline of the main kernel
    main_ms = prof["main_ms"] / args.steps   # every compute launch of a step
    # all pre-pass launches of a step (transposes, re-pitching copies, splits)
    pack_ms = prof["pack_ms"] / args.steps
    peak_tflops = sms * FFMA_PER_SM_PER_CLK * 2 * SM_MAX_MHZ_FALLBACK * 1e6 / 1e12
    peak_meas_clk = (sms * FFMA_PER_SM_PER_CLK * 2 * clk["sm_mhz"] * 1e6 / 1e12
                     if clk.get("sm_mhz") else None)
    if args.path == "ffma" and w.bound == "hbm":
        # HBM: the large operand read once (skinny kernels)
        alg_bytes = 4.0 * (w.M * w.K + w.K * w.N + w.M * w.N * (2 if w.beta != 0 else 1)) * w.batch
        hbm_peak, hsrc = hbm_peak_gbs()
        gbs = alg_bytes / (main_ms * 1e-3) / 1e9 if main_ms > 0 else None
        roofline = {
            "bound": "hbm", "kernel": kernel_text,
            "achieved": round(gbs, 1) if gbs else None, "peak": round(hbm_peak, 1), "unit": "GB/s",
            "frac": round(gbs / hbm_peak, 4) if gbs else None,
            "traffic": load_traffic(w.name),
            **dram_use(load_traffic(w.name), main_ms), "peak_source": hsrc,
            "main_kernel_ms": round(main_ms, 4), "pack_kernels_ms": round(pack_ms, 4),
            "algorithmic_bytes_per_launch": alg_bytes,
        }
    elif args.path == "ffma":
        # FP32 FFMA pipe
        achieved_tflops = w.flops / (main_ms * 1e-3) / 1e12 if main_ms > 0 else None
        f_meas = clk.get("sm_mhz")
        peak_meas = sms * FFMA_PER_SM_PER_CLK * 2 * f_meas * 1e6 / 1e12 if f_meas else None
        roofline = {
            "bound": "alu", "kernel": "sgemm_tma_ffma_kernel",
            "achieved": round(achieved_tflops, 3) if achieved_tflops else None,
            "peak": round(peak_tflops, 3), "unit": "TFLOP/s",
            "frac": round(achieved_tflops / peak_tflops, 4) if achieved_tflops else None,
            "traffic": load_traffic(w.name),
            **dram_use(load_traffic(w.name), main_ms),
            "peak_source": f"derived: {sms} SMs x 128 FFMA/clk x 2 FLOP x 2070 MHz max SM clock",
            "frac_at_measured_clock": (round(achieved_tflops / peak_meas, 4)
                                       if (achieved_tflops and peak_meas) else None),
            "main_kernel_ms": round(main_ms, 4), "pack_kernels_ms": round(pack_ms, 4),
            "algorithmic_flops_per_launch": w.flops,
        }
    else:
        # TF32 tensor pipe: three MMAs per fp32 product
        tpeak, tsrc = tensor_peak_tf32()
        mma_tflops = 3.0 * w.flops / (main_ms * 1e-3) / 1e12 if main_ms > 0 else None
        roofline = {
            "bound": "tensor", "kernel": "sgemm_3xtf32 main kernel (CTA pair or single CTA, chosen per shape)",
            "achieved": round(mma_tflops, 3) if mma_tflops else None,
            "peak": round(tpeak, 3), "unit": "TFLOP/s",
            "frac": round(mma_tflops / tpeak, 4) if mma_tflops else None,
            "traffic": load_traffic(w.name + ":tf32x3"),
            **dram_use(load_traffic(w.name + ":tf32x3"), main_ms), "peak_source": tsrc,
            **probed_mma_fields(mma_tflops, sms, clk.get("sm_mhz")),
            "main_kernel_ms": round(main_ms, 4), "split_kernels_ms": round(pack_ms, 4),
            "algorithmic_flops_per_launch": 3.0 * w.flops,
        }

    # ---- CPU oracle baseline (rank 0 only, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        g, rows, secs = time_oracle_rows(w, A, B, C)
        cpu = {"value": round(g, 3), "unit": "GFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"{rows} full output rows of the {w.M}x{w.N}x{w.K} workload "
                         f"({secs:.1f} s of CPU work)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gflops, 3), "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                       "beta": w.beta, "seed": w.seed,
                       "l2": l2_note(w),
                       "batch": w.batch, "bias": w.bias, "act": w.act,
                       "parallelism": "replicas" if world > 1 else "single_gpu",
                       "kernel": kernel_text},
            "pct_of_ffma_peak": round(100.0 * gflops / world / (peak_tflops * 1e3), 2),
            "pct_of_ffma_peak_at_measured_clock": (
                round(100.0 * gflops / world / (peak_meas_clk * 1e3), 2) if peak_meas_clk else None),
            "per_call": {"pass": "a second pass of the same calls, no profiling events inside them",
                         "median_ms": round(per_call_median, 4), "min_ms": round(per_call_min, 4),
                         "gflops_at_median": round(w.flops / (per_call_median * 1e-3) / 1e9, 3),
                         "gflops_at_min": round(w.flops / (per_call_min * 1e-3) / 1e9, 3),
                         "calls": len(per_call)},
            "sm_count": sms,
            "roofline": roofline,
            "tf32x3": tf32x3,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": int(launches),
            "clocks": {"sm_mhz": clk.get("sm_mhz"), "sm_max_mhz": clk.get("sm_max_mhz"),
                       "reasons": clk.get("reasons"), "samples": clk.get("samples"),
                       "power_w_median": clk.get("power_w_median")},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.oracle_table:
        return run_oracle_table(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
