"""bench.py host logic that needs no GPU: when the committed DRAM-traffic
record applies, and the replica throughput arithmetic."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _records():
    with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
        return json.load(f)


def test_traffic_record_applies_only_to_its_kernel_sources_and_plan():
    rec = _records()["ffma:sq4096_uniform"]
    kernel, grid = rec["kernel"], rec["grid"]
    fresh = rec["csrc_digest"] == bench.kernel_sources_digest("ffma")
    got, note = bench.recorded_traffic(kernel, "sq4096_uniform", "ffma", grid)
    if fresh:
        assert got == rec["dram_bytes_per_launch"] and note
    else:
        assert got is None and "changed" in note
    # Another plan, another grid or another workload never borrows it.
    assert bench.recorded_traffic(kernel + "x", "sq4096_uniform", "ffma", grid)[0] is None
    assert bench.recorded_traffic(kernel, "sq4096_uniform", "ffma", grid + 1)[0] is None
    assert bench.recorded_traffic(kernel, "sq1024_int", "ffma", grid)[0] is None


def test_traffic_record_is_null_once_the_sources_change(monkeypatch):
    rec = _records()["tf32x3:sq4096_uniform"]
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda which="ffma": "0" * 16)
    got, note = bench.recorded_traffic(rec["kernel"], "sq4096_uniform", "tf32x3")
    assert got is None and "changed" in note


def test_recorded_traffic_is_at_least_the_algorithmic_bytes():
    # A launch cannot move less than A and B once and C once (beta == 0).
    n = 4096
    alg = 4 * (n * n + n * n + n * n)
    for key in ("ffma:sq4096_uniform", "tf32x3:sq4096_uniform"):
        assert _records()[key]["dram_bytes_per_launch"] >= 0.9 * alg, key


def test_replica_throughput_counts_every_rank():
    # 2 MNK flops per rank, the slowest rank's time per step.
    one = bench.replica_throughput(2.0 * 4096 ** 3, 2.0, 1)
    assert abs(one - 2.0 * 4096 ** 3 / 2e-3 / 1e9) < 1e-6
    assert abs(bench.replica_throughput(2.0 * 4096 ** 3, 2.0, 8) - 8 * one) < 1e-6


class _RecordingLib:
    """Stands in for the CUDA library: records every entry point touched."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def entry(*args):
            self.calls.append(name)
            return 0
        return entry


def test_3xtf32_leg_never_runs_on_two_or_more_gpus():
    # Its default kernel shares A tiles between CTA pairs by TMA multicast,
    # which is kept out of every run on two or more GPUs.
    from dense_fp32_matrix_strict_gb300 import inputs
    w = inputs.WORKLOADS["sq4096_uniform"]
    call = (w.M, w.N, w.K, 1.0, 1 << 20, w.K, 2 << 20, w.N, 0.0, 3 << 20, w.N, 0)
    args = bench.parse([])
    assert bench.tf32x3_allowed(args, 1)
    assert not bench.tf32x3_allowed(bench.parse(["--no-tf32x3"]), 1)
    for world in (2, 4, 8):
        assert not bench.tf32x3_allowed(args, world)
        lib = _RecordingLib()
        out = bench.measure_3xtf32(args, world, lib, call, torch=None, stream=None, flush=None,
                                   w=w, n=10)
        assert out is None and lib.calls == []
        assert bench.tf32_ceiling(args, world) is None


def test_only_the_guarded_leg_names_the_3xtf32_entry_points():
    # Every use of sgemm_3xtf32* in bench.py sits inside measure_3xtf32, which
    # returns before touching the library unless the run is on one GPU; the
    # per-workload report that also calls it runs only when world == 1.
    import inspect
    src = inspect.getsource(bench)
    leg = inspect.getsource(bench.measure_3xtf32)
    assert src.count('"sgemm_3xtf32"') == leg.count('"sgemm_3xtf32"') > 0
    # The TF32 tensor-core ceiling runs under the same guard.
    assert "tf32x3_allowed(args, world)" in inspect.getsource(bench.tf32_ceiling)
    assert "sgemm_3xtf32_ex" not in src
    run = inspect.getsource(bench.run_ours)
    assert "measure_3xtf32(args, world," in run
    report_at = run.index("workload_report(")
    assert run.rfind("if world == 1:", 0, report_at) >= 0


def test_cpu_baseline_plan_per_workload():
    # The whole problem for the four smaller workloads, a 256-row block plus
    # the sampled entries (extrapolated) for the LLM projection; single-thread
    # rows for 256^3 and 1024^3.
    from dense_fp32_matrix_strict_gb300 import inputs
    whole = [n for n, w in inputs.WORKLOADS.items() if w.flops <= bench.CPU_FULL_LIMIT_FLOP]
    assert whole == ["sq256_uniform", "sq1024_int", "sq4096_uniform",
                     "ragged_4093x5120x1531_normal"]
    assert bench.SINGLE_THREAD_WORKLOADS == ("sq256_uniform", "sq1024_int")
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packAT+sk") == 2
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packATfused+sk") == 1
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packATfused+packB+skfix") == 3
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packATfused+packBTfused+sk") == 1
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packBT+sk") == 2
    assert bench.launches_of("ws_128x128x32_s4_ATtma_Btma+packAT+skfix") == 3
    assert bench.launches_of("ws_128x128x32_s4_Atma_Btma+sk") == 1
    assert bench.launches_of("ws_128x64x32_s4_k2_Axp_Btma") == 1
    assert bench.alg_bytes_of(inputs.WORKLOADS["sq1024_int"]) == 4 * 1024 * 1024 * 4
