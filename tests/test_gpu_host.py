"""sgemm_host: host-resident A, B, C against the CPU oracle.

Covers one block and several (the pipelined path), beta == 0 (C never read)
and beta != 0, leading dimensions wider than the rows with guard values that
must survive, pageable and page-locked buffers, two calls in flight on two
streams, and the integer workload bit for bit.
"""
import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs

pytestmark = pytest.mark.gpu

GUARD = 1.0e30


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    yield


def host(x, ld=None, pin=True):
    """Host tensor view of x with row stride ld; padding holds GUARD."""
    torch = pytest.importorskip("torch")
    rows, cols = x.shape
    ld = max(ld or cols, cols, 1)
    buf = torch.full((max(rows * ld, 1),), GUARD, dtype=torch.float32)
    if pin:
        buf = buf.pin_memory()
    view = buf[:rows * ld].view(rows, ld)[:, :cols]
    if rows and cols:
        view.copy_(torch.from_numpy(np.ascontiguousarray(x)))
    return view, buf


def run(alpha, A, B, beta, C0, lds=(None, None, None), pin=True, stream=None):
    torch = pytest.importorskip("torch")
    hA, _ = host(A, lds[0], pin)
    hB, _ = host(B, lds[1], pin)
    start = C0 if C0 is not None else np.full((A.shape[0], B.shape[1]), np.nan, np.float32)
    hC, bufC = host(start, lds[2], pin)
    sg.sgemm_host_tensors(alpha, hA, hB, beta, hC, stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    sg.check_status()
    ld = max(lds[2] or B.shape[1], B.shape[1], 1)
    pad = bufC.view(-1, ld)[:, B.shape[1]:] if ld > B.shape[1] else None
    guards_ok = pad is None or bool((pad == GUARD).all())
    return hC.numpy().copy(), guards_ok


def check(alpha, A, B, beta, C0, C, exact=False):
    ref, S = oracle.sgemm_ref(alpha, A, B, beta, C0 if beta != 0 else None)
    rep = oracle.check(C, ref, S, A.shape[1], exact=exact)
    assert rep["ok"], rep


def gen(M, N, K, seed, dist="normal"):
    return (inputs.fill(dist, seed, inputs.TID_A, M, K),
            inputs.fill(dist, seed, inputs.TID_B, K, N),
            inputs.fill(dist, seed, inputs.TID_C, M, N))


@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (300, 260, 200),     # one block
                                   (2048, 1536, 1024), (3000, 1100, 1531),   # pipelined
                                   (2100, 2100, 700),                        # B in 4 chunks
                                   (4093, 640, 2100),      # 768, 3 x 1024, ragged 253-row tail
                                   (1100, 2304, 2000)],    # 896 rows in B chunks, 204-row tail
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("beta", [0.0, -1.3])
def test_matches_oracle(shape, beta):
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=M + N + K)
    C, guards = run(0.7, A, B, beta, C0 if beta != 0 else None,
                    lds=(K + 3, N + 5, N + 2))
    assert guards
    check(0.7, A, B, beta, C0, C)


def test_pageable_buffers():
    A, B, C0 = gen(1500, 1400, 1300, seed=5)
    C, guards = run(1.0, A, B, 0.5, C0, pin=False)
    assert guards
    check(1.0, A, B, 0.5, C0, C)


def test_integer_workload_bit_exact():
    w = inputs.WORKLOADS["sq1024_int"]
    A, B, C0 = w.make()
    C, _ = run(w.alpha, A, B, w.beta, C0)
    check(w.alpha, A, B, w.beta, C0, C, exact=True)


def test_alpha_zero_and_k_zero():
    A, B, C0 = gen(64, 48, 32, seed=9)
    C, _ = run(0.0, A, B, 2.0, C0)
    assert np.array_equal(C, (2.0 * C0).astype(np.float32))
    C, _ = run(1.0, A[:, :0], B[:0, :], 0.0, C0)
    assert np.all(C == 0.0)


def test_two_calls_in_flight_on_two_streams():
    torch = pytest.importorskip("torch")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    cases = [gen(2048, 1024, 1024, seed=s) for s in (21, 22)]
    outs = []
    for (A, B, C0), s in zip(cases, (s1, s2)):
        hA, _ = host(A)
        hB, _ = host(B)
        hC, _ = host(C0)
        sg.sgemm_host_tensors(0.7, hA, hB, -1.3, hC, stream=s)
        outs.append(hC)
    s1.synchronize()
    s2.synchronize()
    sg.check_status()
    for (A, B, C0), hC in zip(cases, outs):
        check(0.7, A, B, -1.3, C0, hC.numpy())


def test_rejects_device_tensors():
    torch = pytest.importorskip("torch")
    a = torch.zeros(4, 4, device="cuda")
    with pytest.raises(TypeError):
        sg.sgemm_host_tensors(1.0, a, a, 0.0, a.clone())
