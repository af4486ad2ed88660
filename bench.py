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

``--impl reference`` times that CPU oracle instead (the reference arm): each
step is a bounded row block of the workload.

With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica of the workload (the problem is single-GPU; there is no collective
on the data path); ``value`` is the sum over ranks of the work divided by
the slowest rank's time.
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


def parse():
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
    return ap.parse_args()


# ---------------------------------------------------------------------------
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
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
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
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# Sources each timed kernel's device code is built from (kernel body, PTX
# helpers, the family instantiation). A recorded DRAM-traffic figure is
# reused only while these files are unchanged and the plan (kernel name,
# schedule suffixes, grid) is the one it was captured on.
KERNEL_SOURCES = {
    "ffma": ("sgemm_kernel.cuh", "ptx.cuh", "sgemm_ws_128x128.cu"),
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
    rec = data.get(which + ":" + workload, {})
    if rec.get("kernel") != kernel or rec.get("csrc_digest") != kernel_sources_digest(which):
        return None, None
    if grid is not None and rec.get("grid") != grid:
        return None, None
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
            "sample": f"first {min(rows, w.M)} of {w.M} rows of C (all N={w.N}, K={w.K}), "
                      f"{fl / 1e9:.1f} GFLOP in {dt:.2f} s, double accumulation, OpenMP"}


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


def run_ours(args, w):
    import torch
    import dense_fp32_matrix_strict_gb300 as sg

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
    # the SGEMM kernel, plus the stream-K fixup and any operand packing copy
    launches_per_step = 1 + sum(kernel.count(tag) for tag in ("+sk", "+packA", "+packB"))

    # The timed loop calls the C ABI directly: arguments are marshalled once.
    lib = sg.load()
    call = (w.M, w.N, w.K, float(w.alpha), dA.data_ptr(), w.K, dB.data_ptr(), w.N,
            float(w.beta), dC.data_ptr(), w.N, sh)

    def step():
        if flush is not None:
            flush.zero_()
        rc = lib.sgemm(*call)
        if rc != 0:
            raise sg.SgemmError("sgemm", rc)

    # Measured FFMA ceiling, same process, right before the GEMM.
    clk_peak = ClockSampler(dev).start()
    peak = sg.fp32_peak(target_ms=args.peak_ms)
    peak_clocks = clk_peak.stop()

    for _ in range(max(args.warmup, 3)):
        step()
    sg.check_status()

    # Timed region: K steps between barriers + syncs.
    clk = ClockSampler(dev).start()
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
            rc = lib.sgemm(*call)
            step_ev[i][1].record(stream)
            if rc != 0:
                raise sg.SgemmError("sgemm", rc)
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
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(nev)]
    for i in range(nev):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        rc = lib.sgemm(*call)
        ev[i][1].record(stream)
        if rc != 0:
            raise sg.SgemmError("sgemm", rc)
    torch.cuda.synchronize()
    sg.check_status()
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, world)

    flops = w.flops
    ms_step = total_ms / args.steps
    kernel_ms = statistics.mean(launch_ms)
    value = replica_throughput(flops, ms_step, world)

    # The tcgen05 3xTF32 path, reported separately (same workload, same
    # FP32 error bound, different arithmetic unit).
    tf32x3 = None
    if not args.no_tf32x3:
        call3 = call
        for _ in range(3):
            rc = lib.sgemm_3xtf32(*call3)
            if rc != 0:
                raise sg.SgemmError("sgemm_3xtf32", rc)
        torch.cuda.synchronize()
        n3 = max(10, args.steps // 5)
        x0 = torch.cuda.Event(enable_timing=True)
        x1 = torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for _ in range(n3):
            if flush is not None:
                flush.zero_()
            rc = lib.sgemm_3xtf32(*call3)
            if rc != 0:
                raise sg.SgemmError("sgemm_3xtf32", rc)
        x1.record(stream)
        torch.cuda.synchronize()
        sg.check_status()
        ms3 = max_over_ranks(x0.elapsed_time(x1) / n3, world)
        mp_ = measured_peaks()
        bf16 = float(mp_.get("bf16_tflops") or 1900.0)
        tf32_peak = bf16 * (1.1 / 2.25)      # nominal TF32 : BF16 dense ratio
        tf32_rate = 3.0 * flops / (ms3 * 1e-3) / 1e12
        t3, t3_note = (None, None)
        if os.environ.get("SGEMM_3XTF32_TILE", "128x128c2") == "128x128c2" and w.N > 128:
            t3, t3_note = recorded_traffic("tf32x3_kernel<TcCfg<128,3,2>>", w.name, "tf32x3")
        tf32x3 = {"value": replica_throughput(flops, ms3, world), "unit": "GFLOP/s",
                  "ms_per_step": ms3, "steps": n3,
                  "note": "sgemm_3xtf32: A, B split into TF32 hi/lo, 3 tcgen05 MMAs per product, "
                          "FP32 accumulation in TMEM; same FP32 error bound; times include the "
                          "split pre-passes" + (" and the L2 flush" if flush is not None else ""),
                  "roofline": {"bound": "tensor", "achieved": tf32_rate, "peak": tf32_peak,
                               "unit": "TFLOP/s", "frac": tf32_rate / tf32_peak,
                               "peak_basis": f"measured bf16 {bf16:.1f} TFLOP/s x 1.1/2.25 "
                                             "(nominal TF32:BF16 dense ratio)",
                               "achieved_basis": "3 x 2MNK TF32 FLOP per step / step time",
                               "traffic": t3, "traffic_note": t3_note},
                  "gpu_launches_per_step": 3}

    # Context only, not part of the product: cuBLAS FP32 (torch.addmm with
    # TF32 off) on the same operands, timed the same way on the same stream.
    cublas = None
    if not args.no_cublas:
        prev_tf32 = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        try:
            out = torch.empty_like(dC)
            for _ in range(3):
                torch.addmm(dC, dA, dB, beta=w.beta, alpha=w.alpha, out=out)
            torch.cuda.synchronize()
            nc = max(10, args.steps // 5)
            # As in the timed region: with an L2 flush, events around each
            # call only; otherwise one pair around all of them.
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(nc if flush is not None else 1)]
            if flush is None:
                evs[0][0].record(stream)
            for i in range(nc):
                if flush is not None:
                    flush.zero_()
                    evs[i][0].record(stream)
                torch.addmm(dC, dA, dB, beta=w.beta, alpha=w.alpha, out=out)
                if flush is not None:
                    evs[i][1].record(stream)
            if flush is None:
                evs[0][1].record(stream)
            torch.cuda.synchronize()
            msc = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / nc, world)
            cublas = {"value": replica_throughput(flops, msc, world), "unit": "GFLOP/s",
                      "ms_per_step": msc, "steps": nc,
                      "note": "context only: torch.addmm FP32 with TF32 off (cuBLAS), same "
                              "operands and stream, L2 handled as in the timed region"}
            del out
        finally:
            torch.backends.cuda.matmul.allow_tf32 = prev_tf32

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

    def e2e_step():
        rc = lib.sgemm_host(*hcall)
        if rc != 0:
            raise sg.SgemmError("sgemm_host", rc)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
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
    # The algorithmic minimum of HBM bytes one call moves: A and B read once,
    # C written once (and read once when beta != 0). At the small sizes the
    # path is latency-bound, and the HBM rate says how far from either roof.
    alg_bytes = 4 * (w.M * w.K + w.K * w.N + w.M * w.N * (2 if w.beta != 0 else 1))
    hbm_peak = float(mp.get("hbm_gbs") or 6800.0)
    hbm_achieved = alg_bytes / (kernel_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(w, kernel, grid),
        "frac_of_measured_fp32_ceiling": value / world / peak["gflops"],
        "frac_of_datasheet_fp32": value / world / datasheet,
        "fp32_ceiling": {"measured_gflops": peak["gflops"], "ms": peak["ms"],
                         "clocks": peak_clocks, "datasheet_gflops": datasheet,
                         "datasheet_basis": f"{props.multi_processor_count} SMs x 128 FP32 lanes "
                                            f"x 2 FLOP x {sm_max:.0f} MHz"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": datasheet / 1e3,
                     "unit": "TFLOP/s", "frac": achieved / (datasheet / 1e3),
                     "peak_basis": "FP32 CUDA-core FFMA: SMs x 128 x 2 x max SM clock",
                     "measured_ceiling": peak["gflops"] / 1e3,
                     "frac_of_measured_ceiling": achieved / (peak["gflops"] / 1e3),
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
                              (" + stream-K fixup" if "+sk" in kernel else "") +
                              (" + transposing copy of A" if "+packAT" in kernel else
                               " + packing copy of A" if "+packA" in kernel else "") +
                              (" + transposing copy of B" if "+packBT" in kernel else
                               " + packing copy of B" if "+packB" in kernel else "")) + (
            " (plus one torch L2-flush fill, not ours)" if flush is not None else ""),
    }
    if tf32x3 is not None:
        line["tcgen05_3xtf32"] = tf32x3
    if cublas is not None:
        line["cublas_fp32_context"] = cublas
    if world > 1:
        torch.distributed.destroy_process_group()
    # The CPU oracle baseline is a single-GPU figure: rank 0 times it at N = 1 only.
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, A, B, C0, args.cpu_rows)
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
