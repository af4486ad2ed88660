#!/usr/bin/env python3
"""Benchmark: strict-FP32 SGEMM GFLOP/s on one GB300, as a fraction of the
measured FP32 FFMA ceiling.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one SGEMM call, C = alpha*A*B + beta*C, on the named synthetic
workload (default: M = N = K = 4096, uniform[-1, 1], alpha = 1, beta = 0,
the pages' headline shape). The inputs (A + B + C = 201 MB) are larger than
the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line. ``value`` is GFLOP/s = 2MNK / (device time per step)
with the inputs resident in HBM; ``e2e`` is the same metric when every step
also copies A and B (and C when beta != 0) from pinned host memory and
copies C back. ``roofline`` reports the SGEMM kernel against the FP32
CUDA-core peak (SMs x 128 lanes x 2 FLOP x max SM clock, ``bound: alu``);
``fp32_ceiling`` is the pure-FFMA microbenchmark measured in this run (the
metric's denominator). ``cpu_baseline`` is the double-accumulating CPU
oracle timed on this host on a row block of the same problem.

``tcgen05_3xtf32`` times the separately reported tensor-core entry point
(sgemm_3xtf32: TF32 hi/lo split, three tcgen05 MMAs per product, FP32
accumulation, same error bound) on the same workload, with its own roofline
against the TF32 tensor peak.

``workloads`` (one GPU only) reports all five synthetic workloads the same
way: GFLOP/s, the fractions of the measured ceiling and of the datasheet
rate, the plan, the clocks seen while each was timed, the 3xTF32 path and
cuBLAS FP32 as context, and each workload's CPU oracle timed on this host
(the whole problem; for the 8192 x 14336 x 4096 projection a 256-row block
plus the 65,536 sampled entries, with the full-problem time extrapolated;
single-thread rows for 256^3 and 1024^3). The 256^3 entry also carries the
launch-latency floor (one empty kernel, timed the same way).

``--impl reference`` times that CPU oracle instead (the reference arm): each
step is a bounded row block of the workload.

With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica of the workload (the problem is single-GPU; there is no collective
on the data path); ``value`` is the sum over ranks of the work divided by
the slowest rank's time. The 3xTF32 leg never runs then: its CTA pairs
share A tiles by TMA multicast, which is kept to one-GPU runs.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
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

METRIC = "FP32 SGEMM GFLOP/s (2MNK/t) at 4096³; % of measured GB300 FP32 FMA ceiling"
L2_BYTES = 129 * 1024 * 1024
FP32_LANES_PER_SM = 128


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="sq4096_uniform")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--peak-ms", type=float, default=300.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-tf32x3", action="store_true",
                    help="skip the separately reported tcgen05 3xTF32 measurement")
    ap.add_argument("--no-cublas", action="store_true",
                    help="skip the cuBLAS FP32 context measurement")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="rows of C in the CPU baseline sample (0: sized to ~10 s)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the five-workload report")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
THROTTLE_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


def summarise_clocks(sm, mx, power, reasons, how):
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "sampler": how}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "sm_mhz_min": min(sm),
            "samples": len(sm), "power_w_max": max(power) if power else None,
            "reasons": sorted(reasons), "sampler": how}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (every 200 ms)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, mx, power, reasons = [], [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(THROTTLE_NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return summarise_clocks(sm, mx, power, reasons, "nvidia-smi every 200 ms")


class NvmlSampler:
    """In-process NVML reads of the SM clock, its maximum, board power and
    the clock-event (throttle) reasons every `period_s` (5 ms), so that even
    a timed region of a few tens of milliseconds gets samples. Read-only: it
    changes no setting. Raises OSError from the constructor when NVML or the
    device cannot be found (the caller then falls back to nvidia-smi)."""

    # nvmlClocksEventReason* bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}
    NVML_CLOCK_SM = 1

    def __init__(self, torch_index: int, period_s: float = 0.005):
        import ctypes
        self.ct = ctypes
        self.period = period_s
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None or lib.nvmlInit_v2() != 0:
            raise OSError("NVML unavailable")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if not self._handle(torch_index):
            raise OSError("NVML device not found")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.samples = []
        self.stop_evt = threading.Event()
        self.t = None

    def _handle(self, torch_index):
        import torch
        props = torch.cuda.get_device_properties(torch_index)
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            if self.lib.nvmlDeviceGetHandleByUUID(u.encode(), self.ct.byref(self.h)) == 0:
                return True
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            pci = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), bus,
                                        getattr(props, "pci_device_id", 0))
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(),
                                                        self.ct.byref(self.h)) == 0:
                return True
        return False

    def _one(self):
        ct = self.ct
        sm, mx, pw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(sm)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ct.byref(mx))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw))
        self.reasons_fn(self.h, ct.byref(rs))
        return float(sm.value), float(mx.value), pw.value / 1000.0, int(rs.value)

    def _run(self):
        while not self.stop_evt.is_set():
            v = self._one()
            if v is not None:
                self.samples.append(v)
            self.stop_evt.wait(self.period)

    def start(self):
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()
        return self

    def stop(self):
        self.stop_evt.set()
        if self.t is not None:
            self.t.join(timeout=5)
        v = self._one()          # one reading at the very end as well
        if v is not None:
            self.samples.append(v)
        sm = [x[0] for x in self.samples]
        mx = [x[1] for x in self.samples]
        power = [x[2] for x in self.samples]
        reasons = {n for x in self.samples for n, b in self.BITS.items() if x[3] & b}
        return summarise_clocks(sm, mx, power, reasons, "NVML every 5 ms")


def clock_sampler(torch_index: int):
    """An NVML sampler where NVML is available, else nvidia-smi."""
    try:
        return NvmlSampler(torch_index)
    except (OSError, AttributeError, ImportError):
        return ClockSampler(torch_index)


# ---------------------------------------------------------------------------
# Sources each timed kernel's DRAM traffic depends on (kernel body, PTX
# helpers, the family instantiation, and for the FFMA kernel the planner,
# which sets the tile raster). A recorded DRAM-traffic figure is reused only
# while these files are unchanged and the plan (kernel name, schedule
# suffixes, grid) is the one it was captured on.
# The kernel sgemm_3xtf32's default variant runs on the workloads whose DRAM
# traffic is recorded (CTA pairs on 256 x 256 tiles).
TF32X3_DEFAULT_KERNEL = "tf32x3_pair_kernel"
KERNEL_SOURCES = {
    "ffma": ("sgemm_kernel.cuh", "ptx.cuh", "sgemm_ws_128x128.cu", "sgemm_api.cu"),
    "tf32x3": ("tf32x3.cu", "ptx.cuh"),
}


def kernel_sources_digest(which: str = "ffma") -> str:
    h = hashlib.sha256()
    for name in sorted(KERNEL_SOURCES[which]):
        with open(os.path.join(ROOT, "dense_fp32_matrix_strict_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, which: str = "ffma", grid=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None, None
    with open(path) as f:
        data = json.load(f)
    rec = data.get(which + ":" + workload)
    if rec is None:
        return None, None
    if rec.get("kernel") != kernel or (grid is not None and rec.get("grid") != grid):
        return None, ("the committed ncu record (profiles/ncu_traffic.json) was taken on "
                      "another plan: %s, grid %s" % (rec.get("kernel"), rec.get("grid")))
    if rec.get("csrc_digest") != kernel_sources_digest(which):
        return None, ("the kernel sources changed since the committed ncu record "
                      "(profiles/ncu_traffic.json) was taken")
    return rec.get("dram_bytes_per_launch"), rec.get("note")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
def cpu_oracle_rows(w, A, B, C0, rows: int, nthreads: int = 0):
    """Time the CPU oracle on the first `rows` rows of C; returns (seconds, flops)."""
    import oracle
    r = min(rows, w.M)
    c0 = C0[:r] if w.beta != 0 else None
    t0 = time.perf_counter()
    oracle.sgemm_ref(w.alpha, A[:r], B, w.beta, c0, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, 2.0 * r * w.N * w.K


def cpu_baseline(w, A, B, C0, rows: int):
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    if rows <= 0:
        # Calibrate on a small block, then size the sample to ~10 s.
        probe = max(1, min(w.M, 64))
        dt, fl = cpu_oracle_rows(w, A, B, C0, probe)
        rate = fl / max(dt, 1e-6)
        rows = int(min(w.M, max(1, 10.0 * rate / (2.0 * w.N * w.K))))
    dt, fl = cpu_oracle_rows(w, A, B, C0, rows)
    return {"value": fl / dt / 1e9, "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
            "seconds": dt, "rows": min(rows, w.M),
            "sample": f"first {min(rows, w.M)} of {w.M} rows of C (all N={w.N}, K={w.K}), "
                      f"{fl / 1e9:.1f} GFLOP in {dt:.2f} s, double accumulation, OpenMP"}


# Workloads whose CPU oracle also runs on one thread (the T4 article's CPU
# column is a single-threaded triple loop), and the row block the oracle
# times where the whole problem would take minutes.
SINGLE_THREAD_WORKLOADS = ("sq256_uniform", "sq1024_int")
CPU_FULL_LIMIT_FLOP = 200e9      # above this: a 256-row block + the sampled entries
CPU_BLOCK_ROWS = 256


def workload_cpu_baseline(w, A, B, C0, full=None):
    """The CPU oracle on workload `w`, on this host's cores.

    The whole problem when it is at most 200 GFLOP (``full``: an already
    measured ``cpu_baseline`` dict of the whole problem, reused); otherwise a
    256-row block and the 65,536 seeded sampled entries (plus the last row and
    column) the parity tests check, with the full-problem time extrapolated
    from the block's rate. Single-threaded too for 256^3 and 1024^3."""
    import oracle
    from dense_fp32_matrix_strict_gb300 import inputs
    oracle.build()
    threads = oracle.num_threads()
    if w.flops <= CPU_FULL_LIMIT_FLOP:
        out = dict(full) if full is not None else cpu_baseline(w, A, B, C0, w.M)
        out["sample"] = f"the whole problem ({w.M} x {w.N} x {w.K}), " + out["sample"]
        out["extrapolated"] = False
    else:
        dt, fl = cpu_oracle_rows(w, A, B, C0, CPU_BLOCK_ROWS)
        rows, cols = inputs.sample_entries(w.M, w.N)
        c0 = C0 if w.beta != 0 else None
        t0 = time.perf_counter()
        oracle.sgemm_ref_sampled(w.alpha, A, B, w.beta, c0, rows, cols)
        ds = time.perf_counter() - t0
        fs = 2.0 * w.K * rows.shape[0]
        out = {"value": fl / dt / 1e9, "unit": "GFLOP/s", "cores": threads, "kind": "oracle",
               "seconds": dt, "extrapolated": True,
               "full_problem_seconds_extrapolated": w.flops / (fl / dt),
               "sampled_entries": int(rows.shape[0]), "sampled_seconds": ds,
               "sampled_gflops": fs / ds / 1e9,
               "sample": f"rows 0..{CPU_BLOCK_ROWS - 1} of {w.M} (all N={w.N}, K={w.K}), "
                         f"{fl / 1e9:.1f} GFLOP in {dt:.2f} s; plus the {rows.shape[0]} "
                         f"sampled entries the parity tests check ({ds:.2f} s); the "
                         f"full-problem time ({w.flops / (fl / dt):.0f} s) is extrapolated "
                         f"from the block's rate"}
    if w.name in SINGLE_THREAD_WORKLOADS:
        dt1, fl1 = cpu_oracle_rows(w, A, B, C0, w.M, nthreads=1)
        out["single_thread"] = {"value": fl1 / dt1 / 1e9, "unit": "GFLOP/s", "cores": 1,
                                "seconds": dt1, "ms_per_call": 1e3 * dt1}
    return out


# ---------------------------------------------------------------------------
def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(flops_per_rank: float, ms_per_step: float, world: int) -> float:
    """GFLOP/s of `world` independent replicas: every rank's work divided by
    the slowest rank's time per step (ms_per_step must already be the max)."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, w):
    """Reference arm: the CPU oracle, bounded row blocks of the workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    A, B, C0 = w.make()
    # One step = one row block sized so the whole run stays within minutes.
    probe_dt, probe_fl = cpu_oracle_rows(w, A, B, C0, min(w.M, 16))
    rate = probe_fl / max(probe_dt, 1e-6)
    total_steps = args.steps + args.warmup
    rows = int(max(1, min(w.M, (120.0 / max(total_steps, 1)) * rate / (2.0 * w.N * w.K))))
    for _ in range(args.warmup):
        cpu_oracle_rows(w, A, B, C0, rows)
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, fl = cpu_oracle_rows(w, A, B, C0, rows)
        times.append(dt)
        flops = fl
    total = sum(times)
    value = flops * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, None, None),
        "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: first {rows} of {w.M} rows of C (all N, K)"},
        "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, kernel, grid):
    nbytes = 4 * (w.M * w.K + w.K * w.N + w.M * w.N)
    cfg = {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "beta": w.beta,
           "dist": f"A~{w.dist_a}, B~{w.dist_b}, C0~{w.dist_c}", "seed": w.seed,
           "layout": "row-major, lda=K, ldb=ldc=N",
           "l2": (f"inputs larger than L2 ({nbytes / 2**20:.0f} MiB > 129 MiB), no flush"
                  if nbytes > L2_BYTES else
                  "L2 flushed (258 MB fill) before every step, outside the step's events")}
    if kernel is not None:
        cfg["kernel"] = kernel
        cfg["grid"] = grid
    return cfg


def tf32x3_allowed(args, world: int) -> bool:
    """Whether this run times the 3xTF32 entry point: one-GPU runs only. Its
    default kernel runs CTA pairs that share A tiles by TMA multicast (within
    the calling GPU's own workspace); that load is kept out of every run on
    two or more GPUs, whatever the flags say."""
    return (not args.no_tf32x3) and world == 1


def time_per_call(torch, stream, fn, n: int, flush=None, each: bool = False) -> float:
    """Mean device milliseconds of fn() over n calls on `stream`, by CUDA
    events on that stream: one pair around all n calls, or one pair around
    each call alone when `each` is set or `flush` (a buffer larger than L2)
    is given; the flush buffer is then filled before every call, outside its
    events."""
    if flush is None and not each:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / n


def lib_call(lib, name, args_):
    rc = getattr(lib, name)(*args_)
    if rc != 0:
        import dense_fp32_matrix_strict_gb300 as sg
        raise sg.SgemmError(name, rc)


def tf32_ceiling(args, world):
    """The measured TF32 tensor-core ceiling (back-to-back tcgen05.mma of
    the 3xTF32 kernel's shape on smem-resident operands), one-GPU runs only;
    None where the 3xTF32 leg does not run."""
    if not tf32x3_allowed(args, world):
        return None
    import dense_fp32_matrix_strict_gb300 as sg
    rc, tflops, ms, _ = sg.sgemm_tf32_mma_peak(128, 100.0)
    if rc != sg.SGEMM_OK:
        raise sg.SgemmError("sgemm_tf32_mma_peak", rc)
    return {"tflops": tflops, "ms": ms,
            "basis": "measured: tcgen05.mma.cta_group::1.kind::tf32 M128 N128 K8 back to back "
                     "on shared-memory operands, one CTA per SM (sgemm_tf32_mma_peak)"}


def measure_3xtf32(args, world, lib, call, torch, stream, flush, w, n, peak=None):
    """The separately reported tcgen05 3xTF32 path on the same operands, or
    None where it must not run (see tf32x3_allowed). `peak`: the measured TF32
    ceiling (tf32_ceiling); without it the nominal TF32:BF16 ratio times the
    measured bf16 peak is used, and said so."""
    if not tf32x3_allowed(args, world):
        return None
    import dense_fp32_matrix_strict_gb300 as sg
    for _ in range(3):
        lib_call(lib, "sgemm_3xtf32", call)
    torch.cuda.synchronize()
    ms3 = time_per_call(torch, stream, lambda: lib_call(lib, "sgemm_3xtf32", call), n, flush)
    sg.check_status()
    if peak is not None:
        tf32_peak, peak_basis = peak["tflops"], peak["basis"]
    else:
        mp_ = measured_peaks()
        bf16 = float(mp_.get("bf16_tflops") or 1900.0)
        tf32_peak = bf16 * (1.1 / 2.25)      # nominal TF32 : BF16 dense ratio
        peak_basis = (f"derived: measured bf16 {bf16:.1f} TFLOP/s x 1.1/2.25 "
                      "(nominal TF32:BF16 dense ratio)")
    tf32_rate = 3.0 * w.flops / (ms3 * 1e-3) / 1e12
    t3, t3_note = (None, None)
    if "SGEMM_3XTF32_TILE" not in os.environ:
        # The record names the kernel the default variant ran when it was
        # captured; it is used only while the sources are unchanged.
        t3, t3_note = recorded_traffic(TF32X3_DEFAULT_KERNEL, w.name, "tf32x3")
    return {"value": w.flops / (ms3 * 1e-3) / 1e9, "unit": "GFLOP/s", "ms_per_step": ms3,
            "steps": n,
            "note": "sgemm_3xtf32: A, B split into TF32 hi/lo, 3 tcgen05 MMAs per product, "
                    "FP32 accumulation in TMEM; same FP32 error bound; times include the "
                    "split pre-passes" + ("; L2 flushed before each call, outside its events"
                                          if flush is not None else ""),
            "roofline": {"bound": "tensor", "achieved": tf32_rate, "peak": tf32_peak,
                         "unit": "TFLOP/s", "frac": tf32_rate / tf32_peak,
                         "peak_basis": peak_basis,
                         "achieved_basis": "3 x 2MNK TF32 FLOP per step / step time",
                         "traffic": t3, "traffic_note": t3_note},
            "gpu_launches_per_step": 3}


def measure_cublas(torch, stream, dA, dB, dC, w, n, flush):
    """Context only, not part of the product: cuBLAS FP32 (torch.addmm with
    TF32 off) on the same operands, timed the same way on the same stream."""
    prev_tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        out = torch.empty_like(dC)

        def f():
            torch.addmm(dC, dA, dB, beta=w.beta, alpha=w.alpha, out=out)

        for _ in range(3):
            f()
        torch.cuda.synchronize()
        msc = time_per_call(torch, stream, f, n, flush)
        del out
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev_tf32
    return {"value": w.flops / (msc * 1e-3) / 1e9, "unit": "GFLOP/s", "ms_per_step": msc,
            "steps": n,
            "note": "context only: torch.addmm FP32 with TF32 off (cuBLAS), same operands "
                    "and stream, L2 handled as in the timed region"}


def alg_bytes_of(w) -> int:
    """The algorithmic minimum of HBM bytes one call moves: A and B read
    once, C written once (and read once when beta != 0)."""
    return 4 * (w.M * w.K + w.K * w.N + w.M * w.N * (2 if w.beta != 0 else 1))


def launches_of(kernel: str) -> int:
    """Kernels one sgemm call enqueues: the SGEMM kernel, plus any operand
    packing copy and, when split tiles are finished by a second kernel
    ("+skfix"), that kernel. A stream-K tail finished inside the GEMM kernel
    ("+sk") and copies the GEMM kernel makes itself ("+packATfused",
    "+packBTfused") add no launch."""
    n = 1 + sum(kernel.count(tag) for tag in ("+skfix", "+packA", "+packB"))
    return n - kernel.count("+packATfused") - kernel.count("+packBTfused")


def workload_report(args, lib, torch, stream, dev, w, host, ceiling, datasheet, headline=None,
                    tf32_peak=None):
    """One entry of the five-workload report (GPU side) on the host inputs
    `host` = (A, B, C0). `headline`: the already timed numbers of this
    workload from the main timed region."""
    import dense_fp32_matrix_strict_gb300 as sg
    A, B, C0 = host
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    nbytes = 4 * (w.M * w.K + w.K * w.N + w.M * w.N)
    flush = None
    if nbytes <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    kernel, grid = sg.plan_tensors(w.alpha, dA, dB, w.beta, dC)
    call = (w.M, w.N, w.K, float(w.alpha), dA.data_ptr(), w.K, dB.data_ptr(), w.N,
            float(w.beta), dC.data_ptr(), w.N, stream.cuda_stream)

    def step():
        lib_call(lib, "sgemm", call)

    if headline is None:
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        probe = time_per_call(torch, stream, step, 3, flush)
        n = int(min(400, max(20, 0.15 / max(probe * 1e-3, 1e-7))))
        clk = clock_sampler(dev).start()
        ms = time_per_call(torch, stream, step, n, flush)
        clocks = clk.stop()
        sg.check_status()
    else:
        ms, n, clocks = headline["ms"], headline["steps"], headline["clocks"]
    gflops = w.flops / (ms * 1e-3) / 1e9
    entry = {
        "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha, "beta": w.beta,
        "dist": f"A~{w.dist_a}, B~{w.dist_b}, C0~{w.dist_c}", "seed": w.seed,
        "kernel": kernel, "grid": grid, "gpu_launches_per_call": launches_of(kernel),
        "gflops": gflops, "ms_per_call": ms, "steps": n,
        "frac_of_measured_fp32_ceiling": gflops / ceiling,
        "frac_of_datasheet_fp32": gflops / datasheet,
        "hbm_achieved_gbs": alg_bytes_of(w) / (ms * 1e-3) / 1e9,
        "algorithmic_bytes": alg_bytes_of(w),
        "l2": ("inputs larger than L2, no flush" if flush is None else
               "L2 flushed (258 MB fill) before every call, outside the call's events"),
        "clocks": clocks,
        "parity": ("bit-exact against the oracle (integer inputs)" if w.exact else
                   "every element within 4K 2^-24 S + 1e-6 of the oracle" if w.full_check else
                   "65,536 sampled entries + last row and column within the bound") +
                  " (tests/test_gpu_parity.py, same plan)",
    }
    if w.name == "sq256_uniform":
        # The launch-latency floor, timed the same way (L2 flush, events).
        floor_fn = lambda: lib_call(lib, "sgemm_null_launch", (stream.cuda_stream,))
        for _ in range(3):
            floor_fn()
        entry["latency_floor_ms"] = time_per_call(torch, stream, floor_fn, n, flush)
        entry["latency_floor_note"] = ("one empty kernel (sgemm_null_launch) between the same "
                                       "event pair after the same L2 flush")
    t3 = measure_3xtf32(args, 1, lib, call, torch, stream, flush, w, max(10, n // 4), tf32_peak)
    if t3 is not None:
        entry["tcgen05_3xtf32_gflops"] = t3["value"]
        entry["tcgen05_3xtf32_ms"] = t3["ms_per_step"]
        entry["tcgen05_3xtf32_frac_of_tf32_ceiling"] = t3["roofline"]["frac"]
    if not args.no_cublas:
        cb = measure_cublas(torch, stream, dA, dB, dC, w, max(10, n // 4), flush)
        entry["cublas_fp32_context_gflops"] = cb["value"]
        entry["cublas_fp32_context_ms"] = cb["ms_per_step"]
    del dA, dB, dC, flush
    torch.cuda.empty_cache()
    return entry


def run_ours(args, w):
    import torch
    import dense_fp32_matrix_strict_gb300 as sg
    from dense_fp32_matrix_strict_gb300 import inputs

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    props = torch.cuda.get_device_properties(dev)
    sg.load()
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    A, B, C0 = w.make()
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    nbytes_in = 4 * (w.M * w.K + w.K * w.N + w.M * w.N)
    flush = None
    if nbytes_in <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    kernel, grid = sg.plan_tensors(w.alpha, dA, dB, w.beta, dC)
    launches_per_step = launches_of(kernel)

    # The timed loop calls the C ABI directly: arguments are marshalled once.
    lib = sg.load()
    call = (w.M, w.N, w.K, float(w.alpha), dA.data_ptr(), w.K, dB.data_ptr(), w.N,
            float(w.beta), dC.data_ptr(), w.N, sh)

    def step():
        if flush is not None:
            flush.zero_()
        lib_call(lib, "sgemm", call)

    # Measured FP32 ceiling, same process, right before the GEMM, in both
    # instruction forms (scalar FFMA and the packed FFMA2 the kernel issues);
    # the higher is the metric's denominator.
    clk_peak = clock_sampler(dev).start()
    peak = sg.fp32_peak(target_ms=args.peak_ms, form=sg.SGEMM_PEAK_FFMA)
    peak2 = sg.fp32_peak(target_ms=args.peak_ms, form=sg.SGEMM_PEAK_FFMA2)
    # Context, not a denominator: the kernel's own register outer product
    # without its shared-memory loads (two warps per scheduler).
    peak_outer = sg.fp32_peak(target_ms=args.peak_ms, form=sg.SGEMM_PEAK_OUTER)
    peak_clocks = clk_peak.stop()
    ceiling = max(peak["gflops"], peak2["gflops"])

    for _ in range(max(args.warmup, 3)):
        step()
    sg.check_status()

    # Timed region: K steps between barriers + syncs.
    clk = clock_sampler(dev).start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if flush is None:
        t_start.record(stream)
        for _ in range(args.steps):
            step()
        t_end.record(stream)
    else:
        # Inputs fit in L2: an L2-sized fill runs before every step, outside
        # the step's own pair of events; the step time is the sum of those.
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
        t_start.record(stream)
        for i in range(args.steps):
            flush.zero_()
            step_ev[i][0].record(stream)
            lib_call(lib, "sgemm", call)
            step_ev[i][1].record(stream)
        t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    sg.check_status()
    if flush is None:
        total_ms = t_start.elapsed_time(t_end)
    else:
        total_ms = sum(a.elapsed_time(b) for a, b in step_ev)

    # Launch durations for the roofline: the same call bracketed by CUDA
    # events on the launching stream (covers the SGEMM kernel and, with the
    # stream-K tail, its fixup kernel).
    nev = max(10, min(args.steps, 100))
    kernel_ms = time_per_call(torch, stream, lambda: lib_call(lib, "sgemm", call), nev, flush,
                              each=True)
    sg.check_status()
    total_ms = max_over_ranks(total_ms, world)

    flops = w.flops
    ms_step = total_ms / args.steps
    value = replica_throughput(flops, ms_step, world)

    # The tcgen05 3xTF32 path, reported separately (same workload, same FP32
    # error bound, different arithmetic unit); one-GPU runs only.
    tf32_peak = tf32_ceiling(args, world)
    tf32x3 = measure_3xtf32(args, world, lib, call, torch, stream, flush, w,
                            max(10, args.steps // 5), tf32_peak)
    cublas = None
    if not args.no_cublas:
        cublas = measure_cublas(torch, stream, dA, dB, dC, w, max(10, args.steps // 5), flush)
        cublas["ms_per_step"] = max_over_ranks(cublas["ms_per_step"], world)
        cublas["value"] = replica_throughput(flops, cublas["ms_per_step"], world)

    # End to end through the C ABI with HOST buffers: sgemm_host copies A, B
    # (and C when beta != 0) in and C out, inside the timed region, every
    # step; it overlaps those copies with the GEMMs of row blocks. Each step
    # is a complete call (its copies start after the previous call's work on
    # the stream). C accumulates across steps when beta != 0, as repeated
    # calls in place do.
    hA = torch.from_numpy(A).pin_memory()
    hB = torch.from_numpy(B).pin_memory()
    hOut = torch.from_numpy(C0).pin_memory()
    use_c = w.beta != 0
    h2d = 4 * (w.M * w.K + w.K * w.N + (w.M * w.N if use_c else 0))
    d2h = 4 * w.M * w.N
    hcall = (w.M, w.N, w.K, w.alpha, hA.data_ptr(), w.K, hB.data_ptr(), w.N, w.beta,
             hOut.data_ptr(), w.N, int(stream.cuda_stream))
    for _ in range(3):
        lib_call(lib, "sgemm_host", hcall)
    torch.cuda.synchronize()
    e2e_ms = time_per_call(torch, stream, lambda: lib_call(lib, "sgemm_host", hcall),
                           args.e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, world)
    sg.check_status()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    mp = measured_peaks()
    sm_max = float(mp.get("sm_max_mhz") or 2070.0)
    datasheet = props.multi_processor_count * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e9
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    traffic, traffic_note = recorded_traffic(kernel, w.name, "ffma", grid)
    # At the small sizes the path is latency-bound, and the HBM rate says how
    # far from either roof.
    alg_bytes = alg_bytes_of(w)
    hbm_peak = float(mp.get("hbm_gbs") or 6800.0)
    hbm_achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(w, kernel, grid),
        "frac_of_measured_fp32_ceiling": value / world / ceiling,
        "frac_of_datasheet_fp32": value / world / datasheet,
        "fp32_ceiling": {"measured_gflops": ceiling,
                         "ffma_gflops": peak["gflops"], "ffma_ms": peak["ms"],
                         "ffma2_gflops": peak2["gflops"], "ffma2_ms": peak2["ms"],
                         "basis": "the higher of the scalar FFMA and the packed FFMA2 "
                                  "(fma.rn.f32x2) chain microbenchmarks, this process",
                         "outer_product_gflops": peak_outer["gflops"],
                         "outer_product_note": "context, not a denominator: the 128x128 "
                                               "kernel's 8x8-per-lane packed-FMA outer product "
                                               "with its operands in registers, two warps per "
                                               "scheduler, no shared-memory loads",
                         "clocks": peak_clocks, "datasheet_gflops": datasheet,
                         "datasheet_basis": f"{props.multi_processor_count} SMs x 128 FP32 lanes "
                                            f"x 2 FLOP x {sm_max:.0f} MHz"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": datasheet / 1e3,
                     "unit": "TFLOP/s", "frac": achieved / (datasheet / 1e3),
                     "peak_basis": "FP32 CUDA-core FFMA: SMs x 128 x 2 x max SM clock",
                     "measured_ceiling": ceiling / 1e3,
                     "frac_of_measured_ceiling": achieved / (ceiling / 1e3),
                     "frac_of_outer_product_rate": achieved / (peak_outer["gflops"] / 1e3),
                     "kernel": kernel, "kernel_ms": kernel_ms,
                     "kernel_ms_covers": "every kernel of one sgemm call",
                     "traffic": traffic, "traffic_note": traffic_note,
                     "algorithmic_bytes": alg_bytes, "hbm_achieved_gbs": hbm_achieved,
                     "hbm_peak_gbs": hbm_peak,
                     "hbm_peak_basis": "measured copy bandwidth" if mp.get("hbm_gbs")
                                       else "fallback 6.8 TB/s",
                     "hbm_frac": hbm_achieved / hbm_peak},
        "clocks": clocks,
        "e2e": {"value": replica_throughput(flops, e2e_ms, world), "unit": "GFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "api": "sgemm_host (page-locked host A, B, C; copies overlapped with the "
                       "GEMMs of row blocks inside the call)"},
        "gpu_launches": args.steps * launches_per_step,
        "gpu_launches_note": ("per step: the sgemm kernel" +
                              (" + stream-K fixup kernel" if "+skfix" in kernel else "") +
                              (" (transposed copy of A made inside it)"
                               if "+packATfused" in kernel else
                               " + transposing copy of A" if "+packAT" in kernel else
                               " + packing copy of A" if "+packA" in kernel else "") +
                              (" + transposing copy of B" if "+packBT" in kernel else
                               " + packing copy of B" if "+packB" in kernel else "")) + (
            " (plus one torch L2-flush fill, not ours)" if flush is not None else ""),
    }
    if tf32x3 is not None:
        line["tcgen05_3xtf32"] = tf32x3
    elif world > 1 and not args.no_tf32x3:
        line["tcgen05_3xtf32_skipped"] = ("not run on more than one GPU: its CTA pairs share "
                                          "A tiles by TMA multicast")
    if cublas is not None:
        line["cublas_fp32_context"] = cublas
    if world > 1:
        torch.distributed.destroy_process_group()
    # The CPU oracle baseline and the five-workload report are single-GPU
    # figures: rank 0 takes them at N = 1 only.
    if world == 1:
        del dA, dB, dC, hA, hB, hOut
        torch.cuda.empty_cache()
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, A, B, C0, args.cpu_rows)
        report = {}
        if not args.no_workloads:
            for name, wl in inputs.WORKLOADS.items():
                host = (A, B, C0) if name == w.name else wl.make()
                head = ({"ms": ms_step, "steps": args.steps, "clocks": clocks}
                        if name == w.name else None)
                ent = workload_report(args, lib, torch, stream, dev, wl, host, ceiling,
                                      datasheet, head, tf32_peak)
                if not args.no_cpu_baseline:
                    full = None
                    if name == w.name and line["cpu_baseline"]["rows"] == w.M:
                        full = line["cpu_baseline"]
                    ent["cpu_baseline"] = workload_cpu_baseline(wl, *host, full=full)
                    ent["gpu_over_cpu_oracle"] = ent["gflops"] / ent["cpu_baseline"]["value"]
                report[name] = ent
                del host
        if report:
            line["workloads"] = report
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    from dense_fp32_matrix_strict_gb300 import inputs
    if args.workload not in inputs.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; one of {list(inputs.WORKLOADS)}")
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
