"""sgemm_noalloc: the SGEMM entry point that allocates no device memory.

Callers such as programs whose device memory belongs to another allocator,
or latency-bound paths that may not take an allocator's locks, cannot let the
library call cudaMalloc or a pool allocator. sgemm_noalloc runs the same kernels with the
same schedule but keeps its status word and stream-K partial sums in a fixed
scratch array inside the library.

This test calls it through the C ABI twice in a row (the second call reuses
the scratch the first one left behind) on a problem that takes the stream-K
path. Each result must equal the regular sgemm entry point's bit for bit
(same kernels, same schedule, same summation order) and lie within the
tolerance the parity tests use of the CPU oracle. The scratch status word
must read back clear through sgemm_noalloc_check_status, and the device's
free memory must not shrink between the first call and the second. The file
is collected last, and passes alone in a fresh process as well as after the
other tests.
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
    C_sgemm = d_ref.cpu().numpy()

    # The oracle and the bound of the parity tests, |C - ref| <= 4 K 2^-24 S + 1e-6.
    ref, S = oracle.sgemm_ref(alpha, A, B, beta, C0)
    assert oracle.check(C_sgemm, ref, S, K)["ok"]

    # Every device buffer the calls touch exists before the first call.
    dCs = [torch.from_numpy(C0).cuda() for _ in range(2)]
    torch.cuda.synchronize()
    free = [torch.cuda.mem_get_info()[0]]
    for call, dC in enumerate(dCs):
        rc = sg.sgemm_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                              dC.data_ptr(), N, stream)
        assert rc == sg.SGEMM_OK, (call, rc, sg.sgemm_error_string(rc))
        rc, bits = sg.sgemm_noalloc_check_status(stream)
        assert (rc, bits) == (sg.SGEMM_OK, 0), (call, rc, bits)
        free.append(torch.cuda.mem_get_info()[0])
        C = dC.cpu().numpy()
        assert np.array_equal(C, C_sgemm), (call, int(np.count_nonzero(C != C_sgemm)))
        rep = oracle.check(C, ref, S, K)
        assert rep["ok"], (call, rep)
    # The first call on a device may load the module that holds the 32 MiB
    # scratch array; after that no call takes device memory.
    assert free[0] - free[1] <= (32 << 20) + (2 << 20), free
    assert free[1] - free[2] <= (1 << 20), free
