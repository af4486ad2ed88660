"""Sizes at the edges of what one call takes, against the oracle.

- C with more than 2^31 elements (48,000 x 48,000, 9.2 GB): every offset into
  C, the stream-K partial slots and the transposed copy of A must be 64-bit.
- K = 2^22 with a 3 x 4 (or 3 x 3) C: 131,072 k-tiles, the k-iterations of
  a handful of tiles spread over the SMs in ranges of 4,096.
- 2^21 rows or 2^21 columns with K = 4: 16,384 tiles along one dimension,
  tens of thousands of k-loops of one iteration each.

Inputs come from the seeded generators; the oracle checks every entry where
it finishes in seconds, else the sampled entries plus the whole last row
and column.
"""
import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    return torch


def _gen(M, N, K, seed):
    return (inputs.fill("normal", seed, inputs.TID_A, M, K),
            inputs.fill("normal", seed, inputs.TID_B, K, N),
            inputs.fill("normal", seed, inputs.TID_C, M, N))


def test_c_with_more_than_2_31_elements(torch):
    M = N = 48000
    K = 4
    assert M * N > 2 ** 31
    A = inputs.fill("normal", 41, inputs.TID_A, M, K)
    B = inputs.fill("normal", 41, inputs.TID_B, K, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.empty(M, N, device="cuda", dtype=torch.float32)
    try:
        name, _ = sg.plan_tensors(1.5, dA, dB, 0.0, dC)
        sg.sgemm_tensors(1.5, dA, dB, 0.0, dC)
        sg.check_status()
        rows, cols = inputs.sample_entries(M, N)
        got = dC[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    finally:
        del dC
        torch.cuda.empty_cache()
    ref, S = oracle.sgemm_ref_sampled(1.5, A, B, 0.0, None, rows, cols)
    rep = oracle.check(got, ref, S, K)
    assert rep["ok"], (name, rep)


@pytest.mark.parametrize("N", [4, 3], ids=["B_by_TMA", "B_by_cp_async"])
def test_k_of_2_22(torch, N):
    M, K = 3, 2 ** 22
    A, B, C0 = _gen(M, N, K, seed=42 + N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    name, _ = sg.plan_tensors(0.7, dA, dB, -1.3, dC)
    assert name.endswith("+sk"), name          # a few tiles: the k-iterations are split
    sg.sgemm_tensors(0.7, dA, dB, -1.3, dC)
    sg.check_status()
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    rep = oracle.check(dC.cpu().numpy(), ref, S, K)
    assert rep["ok"], (name, rep)


@pytest.mark.parametrize("shape", [(2 ** 21, 4, 4), (4, 2 ** 21, 4), (2 ** 21, 5, 3)],
                         ids=lambda s: "x".join(map(str, s)))
def test_one_dimension_of_2_21(torch, shape):
    M, N, K = shape
    A, B, C0 = _gen(M, N, K, seed=43)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    name, _ = sg.plan_tensors(1.25, dA, dB, 0.5, dC)
    sg.sgemm_tensors(1.25, dA, dB, 0.5, dC)
    sg.check_status()
    ref, S = oracle.sgemm_ref(1.25, A, B, 0.5, C0)
    rep = oracle.check(dC.cpu().numpy(), ref, S, K)
    assert rep["ok"], (name, rep)
