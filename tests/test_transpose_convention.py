"""The transposition convention of sgemm_ex, checked on the CPU.

The GPU tests hand the oracle op(A) and op(B) as numpy transposes of the
stored matrices. This pins that step to the index formulas the header
states (op(A)(i, k) = A[k * lda + i], op(B)(k, j) = B[j * ldb + k]) by
exact rational arithmetic on flat, padded buffers, so a transposed operand
read the wrong way round cannot pass the GPU tests.
"""
from fractions import Fraction

import numpy as np

import oracle
from dense_fp32_matrix_strict_gb300 import inputs


def flat(x, ld):
    rows, cols = x.shape
    buf = np.full(rows * ld, np.nan, dtype=np.float32)
    for r in range(rows):
        buf[r * ld:r * ld + cols] = x[r]
    return buf


def test_oracle_on_numpy_transposes_matches_the_header_formula():
    M, N, K = 5, 3, 4
    alpha, beta = 0.75, -1.5
    As = inputs.fill("int", 9, inputs.TID_A, K, M)          # A^T stored K x M
    Bs = inputs.fill("int", 9, inputs.TID_B, N, K)          # B^T stored N x K
    C0 = inputs.fill("int", 9, inputs.TID_C, M, N)
    lda, ldb = M + 2, K + 3
    a, b = flat(As, lda), flat(Bs, ldb)
    ref, _ = oracle.sgemm_ref(alpha, np.ascontiguousarray(As.T), np.ascontiguousarray(Bs.T),
                              beta, C0)
    for i in range(M):
        for j in range(N):
            acc = sum(Fraction(float(a[k * lda + i])) * Fraction(float(b[j * ldb + k]))
                      for k in range(K))
            want = Fraction(alpha) * acc + Fraction(beta) * Fraction(float(C0[i, j]))
            assert ref[i, j] == float(want), (i, j)
    # A transpose read as if untransposed gives a different product.
    wrong, _ = oracle.sgemm_ref(alpha, np.ascontiguousarray(As.reshape(M, K)),
                                np.ascontiguousarray(Bs.T), beta, C0)
    assert not np.array_equal(wrong, ref)
