"""sgemm_noalloc: the SGEMM entry point that allocates no device memory.

Callers such as programs whose device memory belongs to another allocator,
or latency-bound paths that may not take an allocator's locks, cannot let the
library call cudaMalloc or a pool allocator. sgemm_noalloc runs the same kernels with the
same schedule but keeps its status word and stream-K partial sums in a fixed
scratch array inside the library.

This test calls it through the C ABI twice in a row (the second call reuses
the scratch the first one left behind) on a problem that takes the stream-K
path, and checks each result against the regular sgemm entry point within
the tolerance the parity tests use. It lives in a file of its own that
pytest collects last, and passes alone in a fresh process as well as after
the other tests.
"""
import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture
def forced_128x128():
    # The 128 x 128 family forced: 72 tiles < 152 SMs, every tile is split.
    assert sg.sgemm_set_config("128x128") == 0
    yield
    sg.sgemm_set_config("auto")


def test_noalloc_matches_sgemm_on_two_calls_in_a_row(forced_128x128):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 1000, 1100, 2000
    alpha, beta = 0.7, -1.3
    A = inputs.fill("normal", 501, inputs.TID_A, M, K)
    B = inputs.fill("normal", 501, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", 501, inputs.TID_C, M, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    stream = torch.cuda.current_stream().cuda_stream

    name, _ = sg.plan_tensors(alpha, dA, dB, beta, torch.empty(M, N, device="cuda"))
    assert name.endswith("+sk"), name      # the scratch-using path

    d_ref = torch.from_numpy(C0).cuda()
    sg.sgemm_tensors(alpha, dA, dB, beta, d_ref)
    sg.check_status()
    C_ref = d_ref.cpu().numpy()

    # The bound of the parity tests, |C - C_ref| <= 4 K 2^-24 S + 1e-6, with
    # S from the CPU oracle.
    _, S = oracle.sgemm_ref(alpha, A, B, beta, C0)
    tol = oracle.error_bound(K, S)

    for call in range(2):
        dC = torch.from_numpy(C0).cuda()
        torch.cuda.synchronize()
        rc = sg.sgemm_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                              dC.data_ptr(), N, stream)
        assert rc == sg.SGEMM_OK, (call, rc, sg.sgemm_error_string(rc))
        torch.cuda.synchronize()
        C = dC.cpu().numpy()
        err = np.abs(C.astype(np.float64) - C_ref.astype(np.float64))
        assert np.all(np.isfinite(C)), call
        assert np.all(err <= tol), (call, float(np.max(err / tol)))
