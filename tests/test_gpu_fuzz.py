"""Seeded random cases across every path the planner can take.

Each case draws a shape (1..700 per dimension, some chosen to cross tile
edges), transposition flags, leading dimensions wider than the rows, base
offsets of 0-3 floats, alpha and beta, and a forced configuration (family,
load modes, A path, schedule), then compares C with the oracle on every
element and checks the guard bands. The draws are fixed by the seed, so a
failure names a reproducible case.
"""
import random

import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu

CONFIGS = ["auto", "auto:dp", "auto:noat", "auto:at", "auto:xp", "128x128", "128x128:xp",
           "128x128:at:dp", "64x64", "64x64:xp", "128x64", "128x64:dp", "128x128:cpasync",
           "64x64:cpasync:dp", "ws_64x128x32_s4", "ws_128x128x32_s3:xp", "ws_128x128x32_s4_l1",
           "ws_128x64x32_s4_k2", "ws_64x64x32_s4_k4:xp", "ws_64x64x32_s4_k2:at",
           "ws_64x64x32_s4_k4:cpasync", "ws_128x64x32_s4_k2:cpasync:dp",
           "ws_64x64x32_s4_k4_c2", "ws_64x64x32_s4_k4_c4:xp", "ws_64x64x32_s4_k4_c4:cpasync"]
EDGES = [1, 2, 3, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257]


def draw(rng):
    def dim():
        return rng.choice(EDGES) if rng.random() < 0.4 else rng.randint(1, 700)
    M, N, K = dim(), dim(), dim()
    ta, tb = rng.random() < 0.3, rng.random() < 0.3
    pad = lambda: rng.choice([0, 0, 1, 3, 4, 8])
    a_cols = M if ta else K
    b_cols = K if tb else N
    lds = (a_cols + pad(), b_cols + pad(), N + pad())
    offs = tuple(rng.choice([0, 0, 1, 2, 3]) for _ in range(3))
    alpha = rng.choice([1.0, 0.7, -1.25])
    beta = rng.choice([0.0, 0.0, 1.0, -0.5])
    cfg = rng.choice(CONFIGS)
    return M, N, K, ta, tb, lds, offs, alpha, beta, cfg


@pytest.mark.parametrize("seed", range(30))
def test_random_cases_match_oracle(seed):
    rng = random.Random(1000 + seed)
    for case in range(12):
        M, N, K, ta, tb, lds, offs, alpha, beta, cfg = draw(rng)
        s = 10_000 * seed + case
        A = inputs.fill("normal", s, inputs.TID_A, M, K)
        B = inputs.fill("normal", s, inputs.TID_B, K, N)
        C0 = inputs.fill("normal", s, inputs.TID_C, M, N)
        As = np.ascontiguousarray(A.T) if ta else A
        Bs = np.ascontiguousarray(B.T) if tb else B
        assert sg.sgemm_set_config(cfg) == 0
        try:
            C, guards, plan = gpu_util.run(alpha, As, Bs, beta, C0 if beta != 0 else None,
                                           lda=lds[0], ldb=lds[1], ldc=lds[2], offsets=offs,
                                           transa=ta, transb=tb)
        finally:
            sg.sgemm_set_config("auto")
        what = (seed, case, M, N, K, ta, tb, lds, offs, alpha, beta, cfg, plan)
        assert guards, what
        ref, S = oracle.sgemm_ref(alpha, A, B, beta, C0 if beta != 0 else None)
        rep = oracle.check(C, ref, S, K)
        assert rep["ok"], (what, rep)
