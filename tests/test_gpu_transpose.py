"""Transposed operands (sgemm_ex, sgemm_3xtf32_ex) against the CPU oracle.

op(A) = A^T means A is stored K x M (element (i, k) of op(A) at
A[k * lda + i]); op(B) = B^T means B is stored N x K. The oracle receives
op(A) and op(B) as plain row-major copies (numpy transposes of the stored
matrices), so it runs its ordinary definition. The bound is the one of the
untransposed path: |C - ref| <= 4 K 2^-24 S + 1e-6, integers bit-exact.
"""
import itertools

import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu

OPS = list(itertools.product([False, True], [False, True]))
OP_IDS = ["NN", "NT", "TN", "TT"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    yield
    sg.sgemm_set_config("auto")


def stored(M, N, K, seed, ta, tb, dist="normal"):
    """Seeded op(A), op(B), C0 and the stored forms of A and B."""
    A = inputs.fill(dist, seed, inputs.TID_A, M, K)
    B = inputs.fill(dist, seed, inputs.TID_B, K, N)
    C0 = inputs.fill(dist, seed, inputs.TID_C, M, N)
    As = np.ascontiguousarray(A.T) if ta else A
    Bs = np.ascontiguousarray(B.T) if tb else B
    return A, B, C0, As, Bs


def check(alpha, A, B, beta, C0, C, exact=False):
    ref, S = oracle.sgemm_ref(alpha, A, B, beta, C0 if beta != 0 else None)
    rep = oracle.check(C, ref, S, A.shape[1], exact=exact)
    assert rep["ok"], rep
    return rep


SHAPES = [(1, 1, 1), (7, 5, 3), (129, 257, 95), (256, 128, 64), (7, 300, 33), (300, 7, 200),
          (513, 130, 1000)]


@pytest.mark.parametrize("ops", OPS, ids=OP_IDS)
@pytest.mark.parametrize("config", ["auto", "128x128", "64x64", "128x64", "128x128:cpasync",
                                    "64x64:dp"])
def test_shapes_match_oracle(ops, config):
    ta, tb = ops
    assert sg.sgemm_set_config(config) == 0
    try:
        for (M, N, K) in SHAPES:
            A, B, C0, As, Bs = stored(M, N, K, 10 + M + N + K, ta, tb)
            C, guards, plan = gpu_util.run(0.7, As, Bs, -1.3, C0, transa=ta, transb=tb)
            assert guards, (config, plan)
            if ta:
                assert "_ATtma_" in plan[0], plan
            if tb:
                assert "+packBT" in plan[0], plan
            check(0.7, A, B, -1.3, C0, C)
    finally:
        sg.sgemm_set_config("auto")


@pytest.mark.parametrize("ops", OPS, ids=OP_IDS)
def test_leading_dims_and_offsets(ops):
    # Stored rows wider than the matrix, bases off 16-byte alignment (offsets
    # of 1-3 floats): a transposed A is then copied before TMA reads it.
    ta, tb = ops
    M, N, K = 300, 260, 200
    A, B, C0, As, Bs = stored(M, N, K, 77, ta, tb)
    for lds, offs in [((None, None, None), (0, 0, 0)),
                      ((As.shape[1] + 3, Bs.shape[1] + 5, N + 7), (1, 2, 3)),
                      ((As.shape[1] + 4, Bs.shape[1] + 8, N + 4), (0, 0, 0))]:
        C, guards, plan = gpu_util.run(1.1, As, Bs, 0.5, C0, lda=lds[0], ldb=lds[1], ldc=lds[2],
                                       offsets=offs, transa=ta, transb=tb)
        assert guards, plan
        if ta:
            aligned = offs[0] == 0 and (lds[0] or As.shape[1]) % 4 == 0
            assert ("+packA" in plan[0]) == (not aligned), plan
        check(1.1, A, B, 0.5, C0, C)


@pytest.mark.parametrize("ops", OPS[1:], ids=OP_IDS[1:])
def test_integer_inputs_bit_exact(ops):
    ta, tb = ops
    A, B, C0, As, Bs = stored(1024, 1024, 1024, 1, ta, tb, dist="int")
    C, guards, _ = gpu_util.run(2.0, As, Bs, -1.0, C0, transa=ta, transb=tb)
    assert guards
    check(2.0, A, B, -1.0, C0, C, exact=True)


@pytest.mark.parametrize("ops", OPS[1:], ids=OP_IDS[1:])
def test_same_bits_as_the_untransposed_call(ops):
    # Same family and schedule: every output sees the same FMA sequence, so
    # op flags on the stored matrices give exactly the bits of the plain call
    # on the transposed copies.
    ta, tb = ops
    M, N, K = 640, 512, 768
    A, B, C0, As, Bs = stored(M, N, K, 5, ta, tb)
    for config in ["128x128", "128x128:dp", "64x64:dp", "128x64:dp"]:
        assert sg.sgemm_set_config(config) == 0
        try:
            C1, _, p1 = gpu_util.run(0.9, A, B, -0.4, C0)
            C2, _, p2 = gpu_util.run(0.9, As, Bs, -0.4, C0, transa=ta, transb=tb)
        finally:
            sg.sgemm_set_config("auto")
        assert p1[1] == p2[1], (p1, p2)
        assert np.array_equal(C1, C2), (config, p1, p2)


SK_SHAPES = [(1024, 1024, 1024), (128, 128, 16384), (333, 4500, 777)]


@pytest.mark.parametrize("ops", OPS[1:], ids=OP_IDS[1:])
@pytest.mark.parametrize("shape", SK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stream_k_tail(ops, shape):
    ta, tb = ops
    M, N, K = shape
    A, B, C0, As, Bs = stored(M, N, K, 31, ta, tb)
    assert sg.sgemm_set_config("128x128") == 0
    try:
        C, guards, plan = gpu_util.run(0.7, As, Bs, -1.3, C0, transa=ta, transb=tb)
    finally:
        sg.sgemm_set_config("auto")
    assert guards and plan[0].endswith("+sk"), plan
    check(0.7, A, B, -1.3, C0, C)


def test_ragged_workload_transposed_both():
    w = inputs.WORKLOADS["ragged_4093x5120x1531_normal"]
    A, B, C0 = w.make()
    As, Bs = np.ascontiguousarray(A.T), np.ascontiguousarray(B.T)
    C, guards, plan = gpu_util.run(w.alpha, As, Bs, w.beta, C0, transa=True, transb=True)
    assert guards, plan
    check(w.alpha, A, B, w.beta, C0, C)


def test_argument_errors():
    torch = pytest.importorskip("torch")
    A = torch.zeros(8, 4, device="cuda")
    C = torch.zeros(4, 4, device="cuda")
    p = A.data_ptr()
    c = C.data_ptr()
    # opa outside {0, 1}
    assert sg.sgemm_ex(2, 0, 4, 4, 8, 1.0, p, 8, p, 4, 0.0, c, 4, 0) == sg.SGEMM_ERR_INVALID_VALUE
    # op(A) = A^T with A stored 8 x 4 means M = 4, K = 8, lda >= M = 4 (ok)
    # and lda = 3 (< M) is rejected.
    B = torch.zeros(8, 4, device="cuda")
    b = B.data_ptr()
    assert sg.sgemm_ex(1, 0, 4, 4, 8, 1.0, p, 4, b, 4, 0.0, c, 4, 0) == sg.SGEMM_OK
    assert sg.sgemm_ex(1, 0, 4, 4, 8, 1.0, p, 3, b, 4, 0.0, c, 4, 0) == sg.SGEMM_ERR_INVALID_VALUE
    # op(B) = B^T with B stored N x K = 4 x 8 needs ldb >= K = 8.
    assert sg.sgemm_ex(0, 1, 4, 4, 8, 1.0, p, 8, b, 7, 0.0, c, 4, 0) == sg.SGEMM_ERR_INVALID_VALUE
    sg.check_status()


@pytest.mark.parametrize("ops", OPS[1:], ids=OP_IDS[1:])
def test_3xtf32_transposed(ops):
    ta, tb = ops
    for (M, N, K) in [(129, 257, 95), (300, 260, 200), (1024, 768, 512)]:
        A, B, C0, As, Bs = stored(M, N, K, 40 + K, ta, tb)
        torch = pytest.importorskip("torch")
        dA = torch.from_numpy(As).cuda()
        dB = torch.from_numpy(Bs).cuda()
        dC = torch.from_numpy(C0).cuda()
        sg.sgemm_3xtf32_tensors(0.7, dA, dB, -1.3, dC, transa=ta, transb=tb)
        sg.check_status()
        check(0.7, A, B, -1.3, C0, dC.cpu().numpy())
