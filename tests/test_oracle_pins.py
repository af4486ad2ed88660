"""The CPU oracle against its pins, and the pins against planted mistakes.

Runs on the CPU only. Every planted mistake lives in a wrapper around the
oracle here, never in the CUDA path.
"""
import numpy as np
import pytest

import oracle
from dense_fp32_matrix_strict_gb300 import inputs
from tests import oracle_pins as pins


def real(alpha, A, B, beta, C0):
    return oracle.sgemm_ref(alpha, A, B, beta, C0)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    pin(real)


def sampled_as_full(alpha, A, B, beta, C0):
    M, N = A.shape[0], B.shape[1]
    r, c = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, S = oracle.sgemm_ref_sampled(alpha, A, B, beta, C0, r.ravel(), c.ravel())
    return ref.reshape(M, N), S.reshape(M, N)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_sampled_oracle_passes_pin(pin):
    pin(sampled_as_full)


# ---- planted mistakes: each must fail at least one pin -------------------

def m_transpose_b(alpha, A, B, beta, C0):
    Bt = np.ascontiguousarray(B.T) if B.shape[0] == B.shape[1] else B[::-1].copy()
    return real(alpha, A, Bt, beta, C0)


def m_drop_last_k(alpha, A, B, beta, C0):
    if A.shape[1] == 0:
        return real(alpha, A, B, beta, C0)
    return real(alpha, np.ascontiguousarray(A[:, :-1]), np.ascontiguousarray(B[:-1]), beta, C0)


def m_beta_sign(alpha, A, B, beta, C0):
    return real(alpha, A, B, -beta, C0)


def m_alpha_on_c(alpha, A, B, beta, C0):
    ref, S = real(1.0, A, B, beta * alpha if alpha != 0 else beta, C0)
    return ref * (alpha if alpha != 0 else 1.0), S


def m_float32_accumulate(alpha, A, B, beta, C0):
    ref, S = real(alpha, A, B, beta, C0)
    if A.shape[1] == 0 or alpha == 0:
        return ref, S
    acc = np.zeros((A.shape[0], B.shape[1]), np.float32)
    for k in range(A.shape[1]):
        acc += np.outer(A[:, k], B[k]).astype(np.float32)
    v = np.float64(np.float32(alpha)) * acc.astype(np.float64)
    if beta != 0:
        v += np.float64(np.float32(beta)) * C0.astype(np.float64)
    return v, S


def m_row_shift(alpha, A, B, beta, C0):
    ref, S = real(alpha, A, B, beta, C0)
    return np.roll(ref, 1, axis=0), S


def m_reads_c_when_beta_zero(alpha, A, B, beta, C0):
    ref, S = real(alpha, A, B, beta, C0)
    if beta == 0 and C0 is not None:
        ref = ref + 0.0 * C0.astype(np.float64)
    return ref, S


def m_magnitude_signed(alpha, A, B, beta, C0):
    ref, S = real(alpha, A, B, beta, C0)
    if A.shape[1] == 0 or alpha == 0:
        return ref, S
    return ref, np.abs(ref)


MUTANTS = [m_transpose_b, m_drop_last_k, m_beta_sign, m_alpha_on_c, m_float32_accumulate,
           m_row_shift, m_reads_c_when_beta_zero, m_magnitude_signed]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m.__name__)
def test_planted_mistake_is_caught(mutant):
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"{mutant.__name__} passed every pin"


def test_sampled_matches_full_bitwise():
    w = inputs.Workload("t", 37, 29, 53, 0.7, -1.3, "normal", "normal", "normal", seed=5)
    A, B, C0 = w.make(lda=60, ldb=31, ldc=30)
    ref, S = oracle.sgemm_ref(w.alpha, A, B, w.beta, C0)
    rows, cols = inputs.sample_entries(w.M, w.N, n=300)
    r2, s2 = oracle.sgemm_ref_sampled(w.alpha, A, B, w.beta, C0, rows, cols)
    assert np.array_equal(r2, ref[rows, cols])
    assert np.array_equal(s2, S[rows, cols])


def test_padding_never_read():
    w = inputs.Workload("t", 9, 7, 5, 1.0, 1.0, "uniform", "uniform", "uniform", seed=6)
    A, B, C0 = w.make(lda=8, ldb=11, ldc=9)        # padding is NaN
    ref, S = oracle.sgemm_ref(w.alpha, A, B, w.beta, C0)
    assert np.all(np.isfinite(ref)) and np.all(np.isfinite(S))


def test_checker_bound_and_exact():
    ref = np.array([[1.0, -2.0]])
    S = np.array([[1.0, 2.0]])
    K = 10
    tol = oracle.error_bound(K, S)
    ok = oracle.check(np.float32(ref + 0.9 * tol), ref, S, K)
    assert ok["ok"], ok
    bad = oracle.check(np.float32(ref + [[0.0, 3 * tol[0, 1]]]), ref, S, K)
    assert not bad["ok"]
    assert oracle.check(np.float32(ref), ref, S, K, exact=True)["ok"]
    assert not oracle.check(np.float32(ref + 1), ref, S, K, exact=True)["ok"]
    nan = oracle.check(np.float32([[np.nan, -2.0]]), ref, S, K)
    assert not nan["ok"]


def test_invalid_args_rejected():
    A = np.zeros((3, 4), np.float32)
    B = np.zeros((5, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.sgemm_ref(1.0, A, B, 0.0, None)
