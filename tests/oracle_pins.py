"""Pins that tie the CPU oracle to facts that do not come from the oracle.

Each ``pin_*`` takes an oracle callable ``fn(alpha, A, B, beta, C0) -> (ref, S)``
and raises ``AssertionError`` when the callable disagrees with:

* ``pin_golden``      the hand-worked example in ``tests/golden/`` (the plain
                      definition C = alpha*A*B + beta*C, "The road to a fast
                      GEMM", section "The problem and the ceiling");
* ``pin_identity``    A = I gives C = B exactly (alpha = 1, beta = 0);
* ``pin_all_ones``    A = B = 1 gives C = K*alpha + beta*C0 exactly;
* ``pin_integer``     exact int64 matrix arithmetic on small integers;
* ``pin_rational``    exact rational arithmetic (``fractions.Fraction``) on
                      tiny real-valued inputs, within the double-precision
                      summation bound (K + 3) * 2^-53 * S;
* ``pin_special``     the BLAS readings: beta == 0 never reads C0, alpha == 0
                      or K == 0 never reads A and B.

``tests/test_oracle_pins.py`` runs every pin on the real oracle and checks
that each planted mistake (a transposed operand, a dropped term, a flipped
sign, float32 accumulation, a wrong index) fails at least one pin.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

from dense_fp32_matrix_strict_gb300 import inputs

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U64 = 2.0 ** -53


def load_golden(name="hand_2x3x2.txt"):
    vals = {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [float(x) for x in rest]
    M, N, K = int(vals["M"][0]), int(vals["N"][0]), int(vals["K"][0])
    f32 = lambda k, r, c: np.array(vals[k], dtype=np.float32).reshape(r, c)
    return dict(M=M, N=N, K=K, alpha=vals["alpha"][0], beta=vals["beta"][0],
                A=f32("A", M, K), B=f32("B", K, N), C0=f32("C0", M, N),
                C=np.array(vals["C"]).reshape(M, N), S=np.array(vals["S"]).reshape(M, N))


def _strided(x, pad):
    """Copy x into a wider NaN-padded buffer and return the strided view."""
    r, c = x.shape
    buf = np.full((r, c + pad), np.nan, dtype=np.float32)
    buf[:, :c] = x
    return buf[:, :c]


def pin_golden(fn):
    g = load_golden()
    ref, S = fn(g["alpha"], g["A"], g["B"], g["beta"], g["C0"])
    assert np.array_equal(ref, g["C"]), (ref, g["C"])
    assert np.array_equal(S, g["S"]), (S, g["S"])


def pin_identity(fn):
    for (n, N) in [(1, 1), (5, 3), (17, 33), (64, 40)]:
        A = np.eye(n, dtype=np.float32)
        B = inputs.fill("normal", 11, inputs.TID_B, n, N)
        C0 = np.full((n, N), np.nan, dtype=np.float32)      # beta == 0: never read
        ref, S = fn(1.0, _strided(A, 3), B, 0.0, C0)
        assert np.array_equal(ref, B.astype(np.float64)), "identity: C != B"
        assert np.array_equal(S, np.abs(B.astype(np.float64))), "identity: S != |B|"


def pin_all_ones(fn):
    for (M, N, K) in [(1, 1, 1), (3, 4, 5), (16, 9, 130), (33, 17, 1000)]:
        A = np.ones((M, K), np.float32)
        B = np.ones((K, N), np.float32)
        C0 = inputs.fill("int", 12, inputs.TID_C, M, N)
        ref, S = fn(2.0, A, _strided(B, 1), -1.0, _strided(C0, 2))
        assert np.array_equal(ref, 2.0 * K - C0.astype(np.float64)), "all-ones: C != 2K - C0"
        assert np.array_equal(S, 2.0 * K + np.abs(C0.astype(np.float64))), "all-ones S"


def pin_integer(fn):
    for (M, N, K, alpha, beta, seed) in [(7, 5, 3, 2.0, -1.0, 21), (40, 24, 70, 3.0, 0.5, 22),
                                         (33, 65, 129, -1.0, 2.0, 23), (16, 16, 16, 1.0, 0.0, 24)]:
        A = inputs.fill("int", seed, inputs.TID_A, M, K)
        B = inputs.fill("int", seed, inputs.TID_B, K, N)
        C0 = inputs.fill("int", seed, inputs.TID_C, M, N)
        ai, bi, ci = (x.astype(np.int64) for x in (A, B, C0))
        prod = ai @ bi                                       # exact integer arithmetic
        mag = np.abs(ai) @ np.abs(bi)
        want = alpha * prod.astype(np.float64) + beta * ci.astype(np.float64)
        want_s = abs(alpha) * mag.astype(np.float64) + abs(beta) * np.abs(ci).astype(np.float64)
        ref, S = fn(alpha, _strided(A, 2), _strided(B, 3), beta, _strided(C0, 1))
        assert np.array_equal(ref, want), "integer pin: value"
        assert np.array_equal(S, want_s), "integer pin: magnitude sum"


def _exact(alpha, A, B, beta, C0):
    """Exact rational value and magnitude sum of every entry."""
    M, K = A.shape
    N = B.shape[1]
    out = np.empty((M, N), dtype=object)
    mag = np.empty((M, N), dtype=object)
    fa, fb = Fraction(float(alpha)), Fraction(float(beta))
    for i in range(M):
        for j in range(N):
            acc, s = Fraction(0), Fraction(0)
            for k in range(K):
                p = Fraction(float(A[i, k])) * Fraction(float(B[k, j]))
                acc += p
                s += abs(p)
            v, m = (fa * acc, abs(fa) * s) if (alpha != 0 and K > 0) else (Fraction(0), Fraction(0))
            if beta != 0:
                c = fb * Fraction(float(C0[i, j]))
                v += c
                m += abs(c)
            out[i, j] = v
            mag[i, j] = m
    return out, mag


def pin_rational(fn):
    cases = [(1, 1, 1, 1.0, 0.0), (2, 3, 5, 0.7, -1.3), (3, 2, 7, -1.1, 0.25),
             (5, 5, 3, 1.0, 1.0), (4, 3, 17, 0.3, -0.9), (2, 2, 31, 1.7, 0.0)]
    for n, (M, N, K, alpha, beta) in enumerate(cases):
        A = inputs.fill("normal", 30 + n, inputs.TID_A, M, K)
        B = inputs.fill("uniform", 30 + n, inputs.TID_B, K, N)
        C0 = inputs.fill("normal", 30 + n, inputs.TID_C, M, N)
        a32, b32 = np.float32(alpha), np.float32(beta)
        ex, exs = _exact(a32, A, B, b32, C0)
        ref, S = fn(alpha, A, B, beta, C0)
        for i in range(M):
            for j in range(N):
                tol = Fraction((K + 3) * U64) * exs[i, j]
                err = abs(Fraction(float(ref[i, j])) - ex[i, j])
                assert err <= tol, f"rational pin {(M, N, K)} at {(i, j)}: err {float(err)}"
                serr = abs(Fraction(float(S[i, j])) - exs[i, j])
                assert serr <= tol, f"rational pin {(M, N, K)} at {(i, j)}: S err {float(serr)}"


def pin_special(fn):
    M, N, K = 6, 5, 4
    A = inputs.fill("uniform", 40, inputs.TID_A, M, K)
    B = inputs.fill("uniform", 40, inputs.TID_B, K, N)
    C0 = inputs.fill("uniform", 40, inputs.TID_C, M, N)
    nanC = np.full((M, N), np.nan, np.float32)
    nanA = np.full((M, K), np.nan, np.float32)
    nanB = np.full((K, N), np.nan, np.float32)
    # beta == 0: C0 is not read, so NaN in C0 must not show.
    ref, _ = fn(1.0, A, B, 0.0, nanC)
    assert np.all(np.isfinite(ref)), "beta == 0 read C0"
    # alpha == 0: A and B are not read; C = beta * C0.
    ref, S = fn(0.0, nanA, nanB, -1.5, C0)
    assert np.array_equal(ref, -1.5 * C0.astype(np.float64)), "alpha == 0"
    assert np.array_equal(S, 1.5 * np.abs(C0.astype(np.float64))), "alpha == 0: S"
    # K == 0: C = beta * C0.
    ref, _ = fn(2.0, np.zeros((M, 0), np.float32), np.zeros((0, N), np.float32), 0.5, C0)
    assert np.array_equal(ref, 0.5 * C0.astype(np.float64)), "K == 0"
    # alpha == 0 and beta == 0: zeros, nothing read.
    ref, _ = fn(0.0, nanA, nanB, 0.0, nanC)
    assert np.array_equal(ref, np.zeros((M, N))), "alpha == beta == 0"


ALL_PINS = [pin_golden, pin_identity, pin_all_ones, pin_integer, pin_rational, pin_special]
