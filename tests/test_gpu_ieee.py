"""Strict IEEE single precision on the FFMA path: no flush of subnormals to
zero, and infinities and NaNs where the definition puts them.

Subnormals: inputs are small integers times 2^-140 (A) and small integers
(B), so every product and every partial sum is a multiple of 2^-140 below
2^-116 and exactly representable; the result must equal the oracle bit for
bit, which a flush-to-zero anywhere (loads, FMAs, stream-K partial sums,
the transposing copy) would break.

Special values: with an infinity or a NaN among the terms of an output's
sum, the IEEE result does not depend on the summation order (no finite
partial sum here comes near overflow), so the kernel must reproduce the
oracle's NaN / +inf / -inf pattern exactly and stay within the usual bound
everywhere else. (The 3xTF32 path splits x into hi + lo, and the lo part of
an infinity is NaN, so that path does not keep infinities; it is not tested
here.)
"""
import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu

CONFIGS = ["auto", "128x128", "128x128:dp", "64x64", "128x64", "128x128:cpasync",
           "128x128:at", "auto:noat"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    yield
    sg.sgemm_set_config("auto")


def subnormal_case(M, N, K, seed):
    A = inputs.fill("int", seed, inputs.TID_A, M, K) * np.float32(2.0 ** -140)
    B = inputs.fill("int", seed, inputs.TID_B, K, N)
    C0 = inputs.fill("int", seed, inputs.TID_C, M, N) * np.float32(2.0 ** -140)
    return A.astype(np.float32), B, C0.astype(np.float32)


@pytest.mark.parametrize("config", CONFIGS)
def test_subnormals_are_not_flushed(config):
    assert np.float32(2.0 ** -140) > 0 and np.float32(2.0 ** -140) < np.finfo(np.float32).tiny
    assert sg.sgemm_set_config(config) == 0
    try:
        for (M, N, K) in [(130, 70, 1000), (300, 260, 200), (1024, 1024, 1024)]:
            A, B, C0 = subnormal_case(M, N, K, seed=M + K)
            assert np.count_nonzero((np.abs(A) < np.finfo(np.float32).tiny) & (A != 0)) > 0
            C, guards, plan = gpu_util.run(1.0, A, B, 1.0, C0)
            assert guards, plan
            ref, S = oracle.sgemm_ref(1.0, A, B, 1.0, C0)
            rep = oracle.check(C, ref, S, K, exact=True)
            assert rep["ok"], (config, plan, rep)
            assert np.count_nonzero(C) > 0.9 * C.size, plan
    finally:
        sg.sgemm_set_config("auto")


def test_subnormals_through_transposed_operands():
    M, N, K = 300, 260, 700
    A, B, C0 = subnormal_case(M, N, K, seed=3)
    As, Bs = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
    C, guards, plan = gpu_util.run(1.0, As, Bs, 1.0, C0, transa=True, transb=True)
    assert guards, plan
    ref, S = oracle.sgemm_ref(1.0, A, B, 1.0, C0)
    assert oracle.check(C, ref, S, K, exact=True)["ok"], plan


def special_case(M, N, K, seed):
    A = inputs.fill("normal", seed, inputs.TID_A, M, K)
    B = inputs.fill("normal", seed, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", seed, inputs.TID_C, M, N)
    A[5, 7] = np.inf            # row 5: +-inf, NaN where B[7, j] == 0
    B[7, 50] = 0.0
    A[9, 3] = np.inf            # row 9: inf - inf = NaN where the signs of
    A[9, 4] = -np.inf           # B[3, j] and B[4, j] agree, else +-inf
    A[11, 2] = np.nan           # row 11: NaN
    B[20, 30] = -np.inf         # column 30: +-inf
    C0[40, 41] = np.inf         # beta * inf
    return A, B, C0


def compare_special(C, ref, S, K):
    nan_c, nan_r = np.isnan(C), np.isnan(ref)
    assert np.array_equal(nan_c, nan_r), np.argwhere(nan_c != nan_r)[:5]
    inf_r = np.isinf(ref)
    assert np.array_equal(np.isinf(C), inf_r)
    assert np.array_equal(C[inf_r], ref[inf_r].astype(np.float32))
    fin = np.isfinite(ref)
    tol = oracle.error_bound(K, S[fin])
    assert np.all(np.abs(C[fin].astype(np.float64) - ref[fin]) <= tol)
    return int(nan_r.sum()), int(inf_r.sum())


@pytest.mark.parametrize("config", CONFIGS)
def test_infinities_and_nans_where_the_definition_puts_them(config):
    M, N, K = 200, 180, 300
    A, B, C0 = special_case(M, N, K, seed=12)
    assert sg.sgemm_set_config(config) == 0
    try:
        C, guards, plan = gpu_util.run(0.5, A, B, 2.0, C0)
    finally:
        sg.sgemm_set_config("auto")
    assert guards, plan
    ref, S = oracle.sgemm_ref(0.5, A, B, 2.0, C0)
    nans, infs = compare_special(C, ref, S, K)
    assert nans >= N and infs >= N // 2, (nans, infs)


def test_special_values_through_stream_k_and_the_transposed_copy():
    # 1024^3 with an infinity: the stream-K partial sums and the transposed
    # copy of A carry it like any other value.
    M = N = K = 1024
    A, B, C0 = special_case(M, N, K, seed=13)
    for config in ["128x128:at", "128x128:noat"]:
        assert sg.sgemm_set_config(config) == 0
        try:
            C, guards, plan = gpu_util.run(1.0, A, B, -1.0, C0)
        finally:
            sg.sgemm_set_config("auto")
        assert guards and plan[0].endswith("+sk"), plan
        ref, S = oracle.sgemm_ref(1.0, A, B, -1.0, C0)
        compare_special(C, ref, S, K)
