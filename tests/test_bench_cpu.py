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
        assert got is None
    # Another plan, another grid or another workload never borrows it.
    assert bench.recorded_traffic(kernel + "x", "sq4096_uniform", "ffma", grid)[0] is None
    assert bench.recorded_traffic(kernel, "sq4096_uniform", "ffma", grid + 1)[0] is None
    assert bench.recorded_traffic(kernel, "sq1024_int", "ffma", grid)[0] is None


def test_traffic_record_is_null_once_the_sources_change(monkeypatch):
    rec = _records()["tf32x3:sq4096_uniform"]
    monkeypatch.setattr(bench, "kernel_sources_digest", lambda which="ffma": "0" * 16)
    assert bench.recorded_traffic(rec["kernel"], "sq4096_uniform", "tf32x3")[0] is None


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
