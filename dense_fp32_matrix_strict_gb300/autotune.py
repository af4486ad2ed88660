"""Per-shape autotuning sweep over the compiled SGEMM kernel configurations.

The best CTA tile, ring depth and schedule depend on the GPU and on the
matrix shape ("The road to a fast GEMM", section "Where to go next",
autotuning; the Tinyforge README's per-size tile sweep and its CSV of
results). This module times every configuration the library offers on each
requested shape and records one CSV row per (shape, configuration):

  * configurations: "auto", "auto" with the transposed copy of A forbidden
    (":noat") and forced (":at"), then every kernel family
    sgemm_config_names lists, each with the stream-K tail allowed and with
    ":dp" (whole tiles only);
  * inputs: seeded uniform [-1, 1) matrices from ``inputs.fill`` (seed 0),
    alpha = 1, beta = 0, dense leading dimensions;
  * timing: CUDA events around each call on the current stream, after
    warm-up calls; when the operands fit in L2 a buffer larger than L2 is
    rewritten before every timed call (outside the events);
  * check (the CSV's ``err_over_bound`` and ``ok``): a self-consistency
    check, not an oracle check. Every configuration's C is compared with
    the "auto" result: both are within 4 K 2^-24 S + 1e-6 of the exact
    product (S = |A| |B| elementwise sums, computed by the library on |A|
    and |B|), so they may differ by at most twice that; a larger difference
    marks the row bad and it is never chosen. A caller may add an
    independent check (``sweep(..., check=f)``): ``f(A, B, C)`` gets the
    host operands and each configuration's result and returns its worst
    error over the bound against a reference of its own; a row is then good
    only if both checks pass, and the value is kept in the row as
    ``ref_err_over_bound`` (not written to the CSV). The package's GPU tests
    pass the CPU oracle this way.

``apply(rows)`` installs the fastest good configuration of each shape with
sgemm_set_shape_config (later sgemm calls on that shape use it while the
global configuration is "auto"); ``load_csv`` reads a saved sweep back.

    python -m dense_fp32_matrix_strict_gb300.autotune \\
        --shapes 4096x4096x4096,4093x5120x1531 --reps 20 --out sweep.csv
"""
from __future__ import annotations

import argparse
import csv
import math
import statistics
import sys
from typing import Iterable

from . import _binding as sg
from . import inputs

FIELDS = ("M", "N", "K", "config", "kernel", "grid", "ms", "gflops", "err_over_bound", "ok",
          "best")
L2_BYTES = 129 * 1024 * 1024


def parse_shapes(text: str) -> list[tuple[int, int, int]]:
    """"MxNxK,MxNxK,..." -> [(M, N, K), ...]."""
    out = []
    for part in text.split(","):
        part = part.strip().lower()
        if not part:
            continue
        dims = part.split("x")
        if len(dims) != 3:
            raise ValueError(f"shape {part!r} is not MxNxK")
        m, n, k = (int(d) for d in dims)
        if min(m, n, k) < 1:
            raise ValueError(f"shape {part!r} has a dimension below 1")
        out.append((m, n, k))
    return out


def all_configs() -> list[str]:
    rc, names = sg.sgemm_config_names()
    if rc != sg.SGEMM_OK:
        raise sg.SgemmError("sgemm_config_names", rc)
    out = ["auto", "auto:noat", "auto:at"]
    for n in names:
        out += [n, n + ":dp"]
    return out


def mark_best(rows: list[dict]) -> list[dict]:
    """Set row["best"] = 1 on the fastest good row of each shape, 0 elsewhere."""
    best = {}
    for r in rows:
        r["best"] = 0
        if not int(r["ok"]) or r["ms"] in ("", None) or not math.isfinite(float(r["ms"])):
            continue
        key = (int(r["M"]), int(r["N"]), int(r["K"]))
        if key not in best or float(r["ms"]) < float(best[key]["ms"]):
            best[key] = r
    for r in best.values():
        r["best"] = 1
    return rows


def write_csv(rows: Iterable[dict], path: str) -> None:
    with open(path, "w", newline="") as f:
        w = csv.DictWriter(f, fieldnames=FIELDS)
        w.writeheader()
        for r in rows:
            w.writerow({k: r.get(k, "") for k in FIELDS})


def load_csv(path: str) -> list[dict]:
    with open(path, newline="") as f:
        return list(csv.DictReader(f))


def best_configs(rows: Iterable[dict]) -> dict[tuple[int, int, int], str]:
    return {(int(r["M"]), int(r["N"]), int(r["K"])): r["config"]
            for r in rows if str(r.get("best", "0")) == "1"}


def apply(rows: Iterable[dict]) -> dict[tuple[int, int, int], str]:
    """Install each shape's best configuration (rows from sweep or load_csv)."""
    chosen = best_configs(rows)
    for (m, n, k), name in chosen.items():
        rc = sg.sgemm_set_shape_config(m, n, k, name)
        if rc != sg.SGEMM_OK:
            raise sg.SgemmError("sgemm_set_shape_config", rc)
    return chosen


def _time_calls(call, reps: int, warmup: int, flush, stream) -> float:
    import torch
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize()
    return statistics.median(x.elapsed_time(y) for x, y in ev)


def _warm_up(lib, stream, seconds: float = 0.1) -> None:
    """Keep the GPU busy for about `seconds` before the first timing, so
    that the first shape is not timed while the clocks ramp up from idle."""
    import time
    import torch
    n = 1024
    A = torch.zeros(n, n, device="cuda")
    C = torch.empty(n, n, device="cuda")
    args = (n, n, n, 1.0, A.data_ptr(), n, A.data_ptr(), n, 0.0, C.data_ptr(), n,
            int(stream.cuda_stream))
    sg.sgemm_set_config("auto")
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(20):
            rc = lib.sgemm(*args)
            if rc != sg.SGEMM_OK:
                raise sg.SgemmError("sgemm", rc)
        torch.cuda.synchronize()


def sweep(shapes, configs=None, reps: int = 20, warmup: int = 3, seed: int = 0,
          log=None, check=None) -> list[dict]:
    """Time every configuration on every shape; returns CSV-ready rows.

    ``check``: optional independent check, ``check(A, B, C) -> worst error
    over bound`` on host float32 arrays (A, B the operands, C the
    configuration's result, alpha = 1, beta = 0)."""
    import torch
    if configs is None:
        configs = all_configs()
    if "auto" not in configs:
        configs = ["auto"] + list(configs)
    stream = torch.cuda.current_stream()
    h = int(stream.cuda_stream)
    lib = sg.load()
    _warm_up(lib, stream)
    rows = []
    try:
        for (M, N, K) in shapes:
            hA = inputs.fill("uniform", seed, inputs.TID_A, M, K)
            hB = inputs.fill("uniform", seed, inputs.TID_B, K, N)
            A = torch.from_numpy(hA).cuda()
            B = torch.from_numpy(hB).cuda()
            C = torch.empty(M, N, device="cuda", dtype=torch.float32)
            flush = None
            if 4 * (M * K + K * N + M * N) <= L2_BYTES:
                flush = torch.empty(2 * L2_BYTES // 4, device="cuda", dtype=torch.float32)
            # S = |A| |B| by the library itself (default configuration).
            sg.sgemm_set_config("auto")
            S = torch.empty_like(C)
            sg.sgemm_tensors(1.0, A.abs(), B.abs(), 0.0, S, stream=stream)
            bound = 2.0 * (4.0 * K * 2.0 ** -24 * S + 1e-6)
            ref = None
            for name in configs:
                rc = sg.sgemm_set_config(name)
                if rc != sg.SGEMM_OK:
                    raise sg.SgemmError("sgemm_set_config", rc)
                call_args = (M, N, K, 1.0, A.data_ptr(), K, B.data_ptr(), N, 0.0, C.data_ptr(),
                             N, h)
                rc, kernel, grid = sg.sgemm_plan(*call_args[:11])
                row = {"M": M, "N": N, "K": K, "config": name, "kernel": kernel, "grid": grid,
                       "ms": "", "gflops": "", "err_over_bound": "", "ok": 0}
                if rc != sg.SGEMM_OK:
                    row["kernel"] = "unavailable: " + sg.sgemm_error_string(rc)
                    rows.append(row)
                    continue

                def call():
                    r = lib.sgemm(*call_args)
                    if r != sg.SGEMM_OK:
                        raise sg.SgemmError("sgemm", r)

                C.fill_(float("nan"))
                call()
                sg.check_status(stream)
                if ref is None:
                    ref = C.clone()
                finite = bool(torch.isfinite(C).all())
                err = float(((C - ref).abs() / bound).max()) if finite else float("inf")
                good = finite and err <= 1.0
                if check is not None:
                    ext = float(check(hA, hB, C.cpu().numpy()))
                    row["ref_err_over_bound"] = ext
                    good = good and ext <= 1.0
                ms = _time_calls(call, reps, warmup, flush, stream)
                sg.check_status(stream)
                row.update(ms=ms, gflops=2.0 * M * N * K / (ms * 1e-3) / 1e9,
                           err_over_bound=err, ok=int(good))
                rows.append(row)
                if log is not None:
                    print(f"{M}x{N}x{K} {name:32s} {kernel:40s} grid {grid:4d} "
                          f"{ms:8.4f} ms {row['gflops']:9.1f} GFLOP/s err/bound {err:.3g}",
                          file=log, flush=True)
            del A, B, C, S, ref, flush, hA, hB
    finally:
        sg.sgemm_set_config("auto")
    return mark_best(rows)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--shapes", required=True, help="MxNxK[,MxNxK...]")
    ap.add_argument("--configs", default=None, help="comma-separated subset (default: all)")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--out", default="sgemm_sweep.csv")
    ap.add_argument("--apply", action="store_true",
                    help="install the winners in this process (useful from Python only)")
    args = ap.parse_args(argv)
    configs = args.configs.split(",") if args.configs else None
    rows = sweep(parse_shapes(args.shapes), configs, args.reps, args.warmup, log=sys.stdout)
    write_csv(rows, args.out)
    for key, name in sorted(best_configs(rows).items()):
        print(f"best {key[0]}x{key[1]}x{key[2]}: {name}")
    if args.apply:
        apply(rows)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
