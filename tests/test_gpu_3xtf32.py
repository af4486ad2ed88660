"""Parity of the tcgen05 3xTF32 entry point (sgemm_3xtf32) with the CPU oracle.

The path is accepted only under the same FP32 bound as the FFMA kernels,
|C - ref| <= 4 K 2^-24 S + 1e-6, and integer-valued inputs (exact in TF32,
with partial sums below 2^24) must come out bit-exact.
"""
import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()


def run_3x(alpha, A, B, beta, C0, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0)):
    import torch
    M, K = A.shape
    N = B.shape[1]
    dA, _, _ = gpu_util.place(A, lda, offsets[0])
    dB, _, _ = gpu_util.place(B, ldb, offsets[1])
    start = C0 if C0 is not None else np.full((M, N), np.nan, np.float32)
    dC, bufC, startC = gpu_util.place(start, ldc, offsets[2])
    sg.sgemm_3xtf32_tensors(alpha, dA, dB, beta, dC)
    sg.check_status()
    torch.cuda.synchronize()
    ok = gpu_util.untouched_outside(bufC, startC, M, N, max(ldc or N, N, 1))
    return dC.cpu().numpy(), ok


SHAPES = [(16, 16, 16), (128, 256, 32), (129, 257, 33), (300, 500, 777), (1, 700, 64),
          (700, 1, 64), (513, 1025, 100), (256, 256, 4096)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes_every_element(shape):
    M, N, K = shape
    A = inputs.fill("normal", 600 + M % 91, inputs.TID_A, M, K)
    B = inputs.fill("normal", 600 + M % 91, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", 600 + M % 91, inputs.TID_C, M, N)
    C, guards = run_3x(0.7, A, B, -1.3, C0)
    assert guards
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    rep = oracle.check(C, ref, S, K)
    assert rep["ok"], rep


@pytest.mark.parametrize("layout", [
    dict(lda=1003, ldb=515, ldc=513, offsets=(1, 2, 3)),
    dict(lda=1000, ldb=512, ldc=512),
], ids=["odd", "padded"])
def test_leading_dims_offsets_and_beta_zero(layout):
    M, N, K = 300, 512, 1000
    A = inputs.fill("uniform", 610, inputs.TID_A, M, K)
    B = inputs.fill("uniform", 610, inputs.TID_B, K, N)
    C, guards = run_3x(1.5, A, B, 0.0, None, **layout)       # beta == 0: C starts NaN
    assert guards and np.all(np.isfinite(C))
    ref, S = oracle.sgemm_ref(1.5, A, B, 0.0, None)
    rep = oracle.check(C, ref, S, K)
    assert rep["ok"], rep


def test_integer_inputs_bit_exact():
    w = inputs.WORKLOADS["sq1024_int"]
    A, B, C0 = w.make()
    C, _ = run_3x(w.alpha, A, B, w.beta, C0)
    ref, S = oracle.sgemm_ref(w.alpha, A, B, w.beta, C0)
    rep = oracle.check(C, ref, S, w.K, exact=True)
    assert rep["ok"], rep


def test_short_k_and_alpha_zero_take_the_ffma_path():
    A = inputs.fill("normal", 611, inputs.TID_A, 64, 5)
    B = inputs.fill("normal", 611, inputs.TID_B, 5, 80)
    C0 = inputs.fill("normal", 611, inputs.TID_C, 64, 80)
    C, _ = run_3x(0.5, A, B, 2.0, C0)
    ref, S = oracle.sgemm_ref(0.5, A, B, 2.0, C0)
    assert oracle.check(C, ref, S, 5)["ok"]
    C, _ = run_3x(0.0, np.full((64, 5), np.nan, np.float32), np.full((5, 80), np.nan, np.float32),
                  2.0, C0)
    assert np.array_equal(C, (np.float32(2.0) * C0).astype(np.float32))


@pytest.mark.parametrize("name", ["sq4096_uniform", "ragged_4093x5120x1531_normal",
                                  "llm_8192x14336x4096"])
def test_workloads_sampled(name):
    w = inputs.WORKLOADS[name]
    A, B, C0 = w.make()
    c0 = C0 if w.beta != 0 else None
    C, guards = run_3x(w.alpha, A, B, w.beta, c0)
    assert guards
    rows, cols = inputs.sample_entries(w.M, w.N)
    ref, S = oracle.sgemm_ref_sampled(w.alpha, A, B, w.beta, c0, rows, cols)
    rep = oracle.check(C[rows, cols], ref, S, w.K)
    assert rep["ok"], rep
    assert np.all(np.isfinite(C))


_SINGLE_CTA_CHILD = r"""
import sys
import numpy as np
import torch
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
M, N, K = (int(v) for v in sys.argv[1:4])
A = inputs.fill("normal", 620, inputs.TID_A, M, K)
B = inputs.fill("normal", 620, inputs.TID_B, K, N)
C0 = inputs.fill("normal", 620, inputs.TID_C, M, N)
dC = torch.from_numpy(C0).cuda()
sg.sgemm_3xtf32_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)
sg.check_status()
np.save(sys.argv[4], dC.cpu().numpy())
"""


@pytest.mark.parametrize("shape", [(300, 640, 500), (513, 1025, 100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cluster_pairs_give_the_single_cta_bits(shape, tmp_path):
    # The default kernel runs CTAs in clusters of two that share A tiles by
    # multicast; each tile still sees the same MMAs in the same order as with
    # one CTA per tile (forced in a child process by SGEMM_3XTF32_TILE).
    import os
    import subprocess
    import sys
    import torch
    M, N, K = shape
    A = inputs.fill("normal", 620, inputs.TID_A, M, K)
    B = inputs.fill("normal", 620, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", 620, inputs.TID_C, M, N)
    dC = torch.from_numpy(C0).cuda()
    sg.sgemm_3xtf32_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)
    sg.check_status()
    pair = dC.cpu().numpy()
    out = str(tmp_path / "single.npy")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, SGEMM_3XTF32_TILE="128x128", PYTHONPATH=root)
    subprocess.run([sys.executable, "-c", _SINGLE_CTA_CHILD, str(M), str(N), str(K), out],
                   check=True, env=env, cwd=root, timeout=300)
    single = np.load(out)
    assert np.array_equal(pair, single)
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    assert oracle.check(pair, ref, S, K)["ok"]


@pytest.mark.parametrize("shape", [(300, 640, 500), (4096, 4096, 256), (1100, 2000, 1531)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cta_pair_mma_gives_the_single_cta_bits(shape, tmp_path):
    # CTA pairs on 256 x 256 tiles (tcgen05.mma.cta_group::2, forced in a
    # child process; the default for large problems) against one CTA per
    # 128 x 128 tile (also forced): every tile sees the same MMAs in the same
    # order, so the bits agree, and both are within the bound of the oracle.
    import os
    import subprocess
    import sys
    M, N, K = shape
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = {}
    for tile in ("256x256", "128x128"):
        out = str(tmp_path / f"{tile}.npy")
        env = dict(os.environ, SGEMM_3XTF32_TILE=tile, PYTHONPATH=root)
        subprocess.run([sys.executable, "-c", _SINGLE_CTA_CHILD, str(M), str(N), str(K), out],
                       check=True, env=env, cwd=root, timeout=300)
        outs[tile] = np.load(out)
    assert np.array_equal(outs["256x256"], outs["128x128"])
    A = inputs.fill("normal", 620, inputs.TID_A, M, K)
    B = inputs.fill("normal", 620, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", 620, inputs.TID_C, M, N)
    rows, cols = inputs.sample_entries(M, N, n=8192)
    ref, S = oracle.sgemm_ref_sampled(0.7, A, B, -1.3, C0, rows, cols)
    assert oracle.check(outs["256x256"][rows, cols], ref, S, K)["ok"]


@pytest.mark.parametrize("shape", [(2304, 2304, 512), (512, 640, 500)],
                         ids=["cta_pairs_256", "tiles_128"])
def test_replays_of_a_captured_graph_give_the_eager_bits(shape):
    # The call's split passes, the MMA kernel launched behind them by
    # programmatic stream serialisation, and its stream-ordered workspace
    # all go into a captured CUDA graph; three replays give the eager bits.
    torch = pytest.importorskip("torch")
    M, N, K = shape
    A = inputs.fill("normal", 412, inputs.TID_A, M, K)
    B = inputs.fill("normal", 412, inputs.TID_B, K, N)
    C0 = inputs.fill("normal", 412, inputs.TID_C, M, N)
    dA, dB, dC0 = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    eager = dC0.clone()
    sg.sgemm_3xtf32_tensors(0.7, dA, dB, -1.3, eager)
    sg.check_status()
    want = eager.cpu().numpy()
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    assert oracle.check(want, ref, S, K)["ok"]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    work = dC0.clone()
    with torch.cuda.graph(g, stream=s):
        sg.sgemm_3xtf32_tensors(0.7, dA, dB, -1.3, work, stream=s)
    for _ in range(3):
        work.copy_(dC0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(work.cpu().numpy(), want)
    sg.check_status()
