"""The transposed copy of a row-major A, and the row-major copy of a
transposed B, made inside the GEMM kernel.

Where "auto" takes the transposed copy of A ("+packAT", the size rule of
tests/test_plan_rule.py) the 128 x 128 kernel makes the copy itself: three
transposer warps per CTA write it unit by unit (BK k-rows x BM columns) in
the order the tiles first need them and release a flag per unit, and the TMA
producer waits for a unit's flag before it loads the unit ("+packATfused").
":atcopy" makes the same copy with a kernel of its own first. Both copies hold
the same values and the GEMM kernel reads them the same way, so the results
must be identical bit for bit, and within the oracle's bound; a call captured
into a CUDA graph makes the copy with its own kernel (a replay would see the
flags of the run before).
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


def run_cfg(cfg, alpha, A, B, beta, C0, **kw):
    assert sg.sgemm_set_config(cfg) == 0
    try:
        return gpu_util.run(alpha, A, B, beta, C0, **kw)
    finally:
        sg.sgemm_set_config("auto")


# Shapes "auto" copies A for: tile rows and k-tiles whole or ragged, lda
# 16-byte aligned or not (A then read by scalar loads), the stream-K tail.
CASES = [
    ((1000, 3000, 4000), {}),
    ((2048, 2048, 8192), {}),
    ((1021, 2600, 3001), {}),
    ((1100, 2900, 2500), {"lda": 2503, "offsets": (1, 0, 0)}),
]


@pytest.mark.parametrize("shape,layout", CASES,
                         ids=["x".join(map(str, s)) + ("_lda" if l else "") for s, l in CASES])
def test_fused_copy_gives_the_separate_copys_bits(shape, layout):
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=1300 + M % 97)
    C1, g1, plan1 = run_cfg("auto", 0.7, A, B, -1.3, C0, **layout)
    C2, g2, plan2 = run_cfg("auto:atcopy", 0.7, A, B, -1.3, C0, **layout)
    assert g1 and g2
    assert "+packATfused" in plan1[0], plan1
    assert "+packAT" in plan2[0] and "+packATfused" not in plan2[0], plan2
    assert plan1[0].replace("+packATfused", "+packAT") == plan2[0] and plan1[1] == plan2[1]
    assert np.array_equal(C1, C2), int(np.count_nonzero(C1 != C2))
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    rep = oracle.check(C1, ref, S, K)
    assert rep["ok"], rep


def test_fused_copy_integers_bit_exact():
    A, B, C0 = gen(1024, 3072, 4096, seed=1310, dist="int")
    C, guards, plan = run_cfg("128x128:at", 2.0, A, B, -1.0, C0)
    assert guards and "+packATfused" in plan[0], plan
    ref, S = oracle.sgemm_ref(2.0, A, B, -1.0, C0)
    assert oracle.check(C, ref, S, 4096, exact=True)["ok"]


def test_workload_4096_takes_the_fused_copy_and_many_calls_agree():
    # The headline shape: the fused copy, and the same bits on calls back to
    # back (each with its own flag value, workspace recycled by the pool).
    torch = pytest.importorskip("torch")
    w = inputs.WORKLOADS["sq4096_uniform"]
    A, B, C0 = w.make()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = [torch.empty(w.M, w.N, device="cuda") for _ in range(4)]
    name, _ = sg.plan_tensors(w.alpha, dA, dB, w.beta, outs[0])
    assert name == "ws_128x128x32_s4_ATtma_Btma+packATfused+sk", name
    for dC in outs:
        sg.sgemm_tensors(w.alpha, dA, dB, w.beta, dC)
    sg.check_status()
    first = outs[0].cpu().numpy()
    for dC in outs[1:]:
        assert np.array_equal(dC.cpu().numpy(), first)
    assert sg.sgemm_set_config("auto:atcopy") == 0
    try:
        ref_c = torch.empty(w.M, w.N, device="cuda")
        sg.sgemm_tensors(w.alpha, dA, dB, w.beta, ref_c)
        sg.check_status()
    finally:
        sg.sgemm_set_config("auto")
    assert np.array_equal(ref_c.cpu().numpy(), first)
    rows, cols = inputs.sample_entries(w.M, w.N)
    ref, S = oracle.sgemm_ref_sampled(w.alpha, A, B, w.beta, None, rows, cols)
    assert oracle.check(first[rows, cols], ref, S, w.K)["ok"]


def test_captured_call_copies_with_its_own_kernel():
    # Captured into a graph the call makes the copy with its own kernel; the
    # replays give the eager (fused) call's bits.
    torch = pytest.importorskip("torch")
    M, N, K = 2048, 2048, 8192
    A, B, C0 = gen(M, N, K, seed=1320)
    dA, dB, dC0 = (torch.from_numpy(x).cuda() for x in (A, B, C0))
    eager = dC0.clone()
    name, _ = sg.plan_tensors(0.7, dA, dB, -1.3, eager)
    assert "+packATfused" in name, name
    sg.sgemm_tensors(0.7, dA, dB, -1.3, eager)
    sg.check_status()
    want = eager.cpu().numpy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    work = dC0.clone()
    with torch.cuda.graph(g, stream=s):
        sg.sgemm_tensors(0.7, dA, dB, -1.3, work, stream=s)
    for _ in range(3):
        work.copy_(dC0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(work.cpu().numpy(), want)
    sg.check_status()


def test_two_streams_concurrently():
    # Two fused calls at a time on two streams with no ordering between them:
    # each has its own workspace, flags and flag value; a kernel whose CTAs
    # are not all on the GPU yet (the other kernel still holds SMs) waits for
    # them within its bounded waits. Three rounds, every result checked.
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 3000, 4000
    A1, B1, C1 = gen(M, N, K, seed=1330)
    A2, B2, C2 = gen(M, N, K, seed=1331)
    d = [torch.from_numpy(x).cuda() for x in (A1, B1, C1, A2, B2, C2)]
    name, _ = sg.plan_tensors(0.7, d[0], d[1], -1.3, d[2])
    assert "+packATfused" in name, name
    want1, _, _ = run_cfg("auto:atcopy", 0.7, A1, B1, -1.3, C1)
    want2, _, _ = run_cfg("auto:atcopy", 0.7, A2, B2, -1.3, C2)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            c1 = d[2].clone()
            sg.sgemm_tensors(0.7, d[0], d[1], -1.3, c1, stream=s1)
        with torch.cuda.stream(s2):
            c2 = d[5].clone()
            sg.sgemm_tensors(0.7, d[3], d[4], -1.3, c2, stream=s2)
        torch.cuda.synchronize()
        sg.check_status()
        assert np.array_equal(c1.cpu().numpy(), want1)
        assert np.array_equal(c2.cpu().numpy(), want2)


# (M, N, K, transa, transb): a transposed B whose row-major copy the kernel
# makes itself, beside the transposed copy of a row-major A (N, T) or with A
# given transposed and read in place (T, T); ragged edges in the last three,
# and in the last two a K that is not a multiple of 4, so that the rows of
# the stored B (and in the last of A) are not 16-byte aligned and the units
# are read by scalar loads.
B_CASES = [(4096, 2048, 4096, False, True), (2048, 2048, 2048, True, True),
           (2000, 2100, 1900, True, True), (2000, 2100, 1531, True, True),
           (4093, 2560, 1531, False, True)]


@pytest.mark.parametrize("M,N,K,ta,tb", B_CASES,
                         ids=["x".join(map(str, c[:3])) + ("_T" if c[3] else "_N") + "T"
                              for c in B_CASES])
def test_fused_copy_of_a_transposed_b(M, N, K, ta, tb):
    A = inputs.fill("normal", 1340, inputs.TID_A, *((K, M) if ta else (M, K)))
    B = inputs.fill("normal", 1340, inputs.TID_B, *((N, K) if tb else (K, N)))
    C0 = inputs.fill("normal", 1340, inputs.TID_C, M, N)
    C1, g1, plan1 = run_cfg("auto", 0.7, A, B, -1.3, C0, transa=ta, transb=tb)
    C2, g2, plan2 = run_cfg("auto:atcopy", 0.7, A, B, -1.3, C0, transa=ta, transb=tb)
    assert g1 and g2
    assert "+packBTfused" in plan1[0], plan1
    assert ("+packATfused" in plan1[0]) == (not ta), plan1
    assert "+packBT" in plan2[0] and "fused" not in plan2[0], plan2
    assert np.array_equal(C1, C2), int(np.count_nonzero(C1 != C2))
    opA = A.T if ta else A
    opB = B.T if tb else B
    ref, S = oracle.sgemm_ref(0.7, np.ascontiguousarray(opA), np.ascontiguousarray(opB), -1.3, C0)
    assert oracle.check(C1, ref, S, K)["ok"]


# Stored operands with padded rows (NaN between them, which must never reach C)
# and base addresses off the 16-byte grid, so both fused copies read their
# units by scalar loads; C padded too, its guard bands checked.
PADDED_B_CASES = [
    ((2000, 2100, 1531, True, True), dict(lda=2004, ldb=1536, offsets=(0, 1, 0))),
    ((4093, 2560, 1531, False, True), dict(lda=1533, ldb=1534, ldc=2564, offsets=(1, 2, 3))),
]


@pytest.mark.parametrize("case,layout", PADDED_B_CASES,
                         ids=["x".join(map(str, c[:3])) + ("_T" if c[3] else "_N") + "T"
                              for c, _ in PADDED_B_CASES])
def test_fused_copies_of_padded_unaligned_operands(case, layout):
    M, N, K, ta, tb = case
    A = inputs.fill("normal", 1350, inputs.TID_A, *((K, M) if ta else (M, K)))
    B = inputs.fill("normal", 1350, inputs.TID_B, *((N, K) if tb else (K, N)))
    C0 = inputs.fill("normal", 1350, inputs.TID_C, M, N)
    C1, g1, plan1 = run_cfg("auto", 0.7, A, B, -1.3, C0, transa=ta, transb=tb, **layout)
    C2, g2, plan2 = run_cfg("auto:atcopy", 0.7, A, B, -1.3, C0, transa=ta, transb=tb, **layout)
    assert g1 and g2
    assert "+packBTfused" in plan1[0], plan1
    assert ("+packATfused" in plan1[0]) == (not ta), plan1
    assert "fused" not in plan2[0], plan2
    assert np.array_equal(C1, C2), int(np.count_nonzero(C1 != C2))
    opA = A.T if ta else A
    opB = B.T if tb else B
    ref, S = oracle.sgemm_ref(0.7, np.ascontiguousarray(opA), np.ascontiguousarray(opB), -1.3, C0)
    assert oracle.check(C1, ref, S, K)["ok"]
