"""The autotuning sweep on the GPU: every configuration it times must agree
with the default one within the FP32 bound (the sweep's own self-consistency
column) and with the CPU oracle on sampled entries (an independent check the
test hands the sweep), and the per-shape rule it installs must change the
plan of that shape only."""
import numpy as np
import pytest

import oracle
from dense_fp32_matrix_strict_gb300 import inputs

import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import autotune

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    sg.sgemm_clear_shape_configs()
    yield
    sg.sgemm_clear_shape_configs()
    sg.sgemm_set_config("auto")


def _plan(M, N, K):
    import torch
    A = torch.empty(M, K, device="cuda")
    B = torch.empty(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    return sg.plan_tensors(1.0, A, B, 0.0, C)[0]


def oracle_check(A, B, C):
    """Worst |C - ref| / bound over 4,096 seeded entries (plus the last row
    and column) against the CPU oracle, alpha = 1, beta = 0."""
    M, K = A.shape
    N = B.shape[1]
    rows, cols = inputs.sample_entries(M, N, n=4096)
    ref, S = oracle.sgemm_ref_sampled(1.0, A, B, 0.0, None, rows, cols)
    got = C[rows, cols].astype(np.float64)
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(np.max(np.abs(got - ref) / oracle.error_bound(K, S)))


def test_sweep_rows_are_checked_and_one_is_best(tmp_path):
    shapes = [(300, 260, 200), (1024, 768, 512)]
    configs = autotune.all_configs()
    rows = autotune.sweep(shapes, configs, reps=2, warmup=1, check=oracle_check)
    assert len(rows) == len(shapes) * len(configs)
    for r in rows:
        assert r["ok"] == 1, r
        assert r["ms"] > 0 and r["err_over_bound"] <= 1.0
        # every configuration against the CPU oracle, not only against "auto"
        assert r["ref_err_over_bound"] <= 1.0, r
    for s in shapes:
        assert sum(r["best"] for r in rows if (r["M"], r["N"], r["K"]) == s) == 1
    p = tmp_path / "sweep.csv"
    autotune.write_csv(rows, str(p))
    assert autotune.best_configs(autotune.load_csv(str(p))) == autotune.best_configs(rows)
    # The sweep leaves the global configuration at "auto".
    assert sg.sgemm_set_config("auto") == 0


def test_shape_rule_changes_only_its_shape():
    # 2048 x 2048 x 1024 runs the 128 x 128 family with the stream-K tail
    # by default.
    base = _plan(2048, 2048, 1024)
    other = _plan(2048, 2048, 1056)
    assert base.startswith("ws_128x128x32_s4_") and base.endswith("+sk")
    assert sg.sgemm_set_shape_config(2048, 2048, 1024, "64x64:dp") == 0
    try:
        assert _plan(2048, 2048, 1024).startswith("ws_64x64x32_s4_")
        assert "+sk" not in _plan(2048, 2048, 1024)
        assert _plan(2048, 2048, 1056) == other
        # A global configuration other than "auto" takes precedence.
        assert sg.sgemm_set_config("ws_128x128x32_s6") == 0
        assert _plan(2048, 2048, 1024).startswith("ws_128x128x32_s6_")
        assert sg.sgemm_set_config("auto") == 0
        assert _plan(2048, 2048, 1024).startswith("ws_64x64x32_s4_")
    finally:
        sg.sgemm_set_config("auto")
        sg.sgemm_set_shape_config(2048, 2048, 1024, "auto")
    assert _plan(2048, 2048, 1024) == base


def test_apply_installs_the_winners():
    rows = autotune.mark_best([
        {"M": 333, "N": 444, "K": 555, "config": "ws_128x128x32_s3:dp", "ms": 1.0, "ok": 1},
        {"M": 333, "N": 444, "K": 555, "config": "auto", "ms": 2.0, "ok": 1},
    ])
    try:
        assert autotune.apply(rows) == {(333, 444, 555): "ws_128x128x32_s3:dp"}
        assert _plan(333, 444, 555).startswith("ws_128x128x32_s3_")
    finally:
        sg.sgemm_clear_shape_configs()
