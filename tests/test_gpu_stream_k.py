"""The stream-K tail's two ways of finishing a split tile, on the GPU.

By default the CTA that holds a split tile's first k-segment finishes it
inside the GEMM kernel: the CTAs holding the later segments leave their raw
sums in workspace slots and set a flag each, and the finishing CTA waits for
the flags, adds the slots in k order and runs the epilogue. ":fixup" selects
the older way, a second kernel that adds the same slots in the same order.
Both must give the same bits (same sums, same order), match the oracle, and
survive replays of a captured CUDA graph (the finishing CTA resets the flags
it consumed, so a replay with the same flag value never reads stale slots).
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
    sg.sgemm_set_config("auto")
    yield
    sg.sgemm_set_config("auto")


def gen(M, N, K, seed, dist="normal"):
    return (inputs.fill(dist, seed, inputs.TID_A, M, K),
            inputs.fill(dist, seed, inputs.TID_B, K, N),
            inputs.fill(dist, seed, inputs.TID_C, M, N))


def run_cfg(cfg, alpha, A, B, beta, C0):
    assert sg.sgemm_set_config(cfg) == 0
    try:
        return gpu_util.run(alpha, A, B, beta, C0)
    finally:
        sg.sgemm_set_config("auto")


# (family, shape): shapes whose last wave is split, for the 128 x 128 tile,
# the 128 x 64 tile in two k-groups, the 64 x 64 tile in four k-groups and
# cp.async loads; tiles split into 2, 3 or dozens of segments.
CASES = [
    ("128x128", (1000, 1100, 2000)),          # 72 tiles < 152 CTAs: every tile split
    ("128x128", (1024, 1024, 1024)),          # 64 tiles of 32 k-tiles, ~2.4 segments each
    ("128x128", (512, 5504, 96)),             # one full wave + a 20-tile tail
    ("128x128", (130, 70, 8400)),             # few tiles, many segments each
    ("128x128:cpasync", (333, 4500, 777)),    # cp.async producers, ragged edges
    ("ws_128x64x32_s4_k2", (1024, 1024, 1024)),
    ("ws_64x64x32_s4_k4", (256, 256, 8192)),
    ("auto", (2048, 2048, 8192)),             # transposed copy of A made in the kernel + tail
]


@pytest.mark.parametrize("cfg,shape", CASES, ids=lambda x: x if isinstance(x, str)
                         else "x".join(map(str, x)))
def test_in_kernel_finish_matches_fixup_kernel_bitwise_and_oracle(cfg, shape):
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=900 + M % 101 + K % 13)
    C1, g1, plan1 = run_cfg(cfg, 0.7, A, B, -1.3, C0)
    C2, g2, plan2 = run_cfg(cfg + ":fixup", 0.7, A, B, -1.3, C0)
    assert g1 and g2
    assert plan1[0].endswith("+sk"), plan1
    assert plan2[0].endswith("+skfix"), plan2
    assert plan1[0][:-3] == plan2[0][:-6] and plan1[1] == plan2[1]
    assert np.array_equal(C1, C2), int(np.count_nonzero(C1 != C2))
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    rep = oracle.check(C1, ref, S, K)
    assert rep["ok"], rep


def test_in_kernel_finish_integers_bit_exact():
    A = inputs.fill("int", 7, inputs.TID_A, 1024, 1024)
    B = inputs.fill("int", 7, inputs.TID_B, 1024, 1024)
    C0 = inputs.fill("int", 7, inputs.TID_C, 1024, 1024)
    C, guards, plan = run_cfg("128x128", 2.0, A, B, -1.0, C0)
    assert guards and plan[0].endswith("+sk"), plan
    ref, S = oracle.sgemm_ref(2.0, A, B, -1.0, C0)
    assert oracle.check(C, ref, S, 1024, exact=True)["ok"]


def test_many_calls_in_a_row_reuse_no_stale_flag():
    # Back-to-back calls on one stream (each with its own flag value, the
    # workspace recycled by the pool) and then one more: all equal.
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 1100, 2000
    A, B, C0 = gen(M, N, K, seed=910)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    assert sg.sgemm_set_config("128x128") == 0
    try:
        outs = [torch.from_numpy(C0).cuda() for _ in range(8)]
        for dC in outs:
            sg.sgemm_tensors(0.7, dA, dB, -1.3, dC)
        sg.check_status()
        first = outs[0].cpu().numpy()
        for dC in outs[1:]:
            assert np.array_equal(dC.cpu().numpy(), first)
    finally:
        sg.sgemm_set_config("auto")
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    assert oracle.check(first, ref, S, K)["ok"]


def test_graph_replays_reset_the_flags():
    # A captured launch keeps its flag value on every replay; the finishing
    # CTAs reset the flags they consumed, so each replay waits for its own
    # slots. Three replays must give the eager call's bits.
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 1100, 2000
    A, B, C0 = gen(M, N, K, seed=911)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    assert sg.sgemm_set_config("128x128") == 0
    try:
        eager = dC.clone()
        sg.sgemm_tensors(0.7, dA, dB, -1.3, eager)
        sg.check_status()
        want = eager.cpu().numpy()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        work = dC.clone()
        with torch.cuda.graph(g):
            sg.sgemm_tensors(0.7, dA, dB, -1.3, work)
        for _ in range(3):
            work.copy_(dC)
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(work.cpu().numpy(), want)
        sg.check_status()
    finally:
        sg.sgemm_set_config("auto")
