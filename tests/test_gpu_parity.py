"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Real-valued inputs: every element within |C - ref| <= 4 K 2^-24 S + 1e-6
(S = |alpha| sum_k |a_ik b_kj| + |beta c_ij|). Integer-valued inputs: bit-exact.
Small shapes are checked on every element; the full workloads on every
element where the oracle finishes in seconds, else on 65,536 seeded entries
plus the whole last row and column.
"""
import re

import numpy as np
import pytest

import oracle
import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

pytestmark = pytest.mark.gpu

CONFIGS = ["auto", "128x128", "64x64", "128x128:cpasync", "64x64:cpasync"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    yield
    sg.sgemm_set_config("auto")


@pytest.fixture
def config(request):
    name = getattr(request, "param", "auto")
    assert sg.sgemm_set_config(name) == 0
    yield name
    sg.sgemm_set_config("auto")


def gen(M, N, K, seed, dist="normal"):
    A = inputs.fill(dist, seed, inputs.TID_A, M, K)
    B = inputs.fill(dist, seed, inputs.TID_B, K, N)
    C0 = inputs.fill(dist, seed, inputs.TID_C, M, N)
    return A, B, C0


def check_full(alpha, A, B, beta, C0, C, exact=False):
    ref, S = oracle.sgemm_ref(alpha, A, B, beta, C0 if beta != 0 else None)
    rep = oracle.check(C, ref, S, A.shape[1], exact=exact)
    assert rep["ok"], rep
    return rep


SHAPES = [(1, 1, 1), (2, 3, 5), (7, 5, 3), (31, 33, 17), (64, 64, 32), (127, 129, 33),
          (128, 128, 32), (129, 127, 31), (255, 257, 63), (300, 200, 100), (513, 130, 1000),
          (1, 1000, 7), (1000, 1, 7), (65, 64, 1), (64, 65, 2), (256, 256, 256)]


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_every_element(config, shape):
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=100 + M + 7 * N + 13 * K)
    C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
    assert guards, "wrote outside C"
    check_full(0.7, A, B, -1.3, C0, C)
    if config.endswith("cpasync"):
        assert "Acp_Bcp" in plan[0], plan


@pytest.mark.parametrize("config", CONFIGS, indirect=True)
@pytest.mark.parametrize("layout", [
    dict(lda=None, ldb=None, ldc=None, offsets=(0, 0, 0)),       # dense, 16-byte aligned
    dict(lda=37, ldb=70, ldc=71, offsets=(0, 0, 0)),             # unaligned leading dims
    dict(lda=40, ldb=72, ldc=72, offsets=(1, 2, 3)),             # aligned lds, shifted bases
    dict(lda=36, ldb=68, ldc=68, offsets=(4, 8, 0)),             # padded, 16-byte aligned
], ids=["dense", "odd_ld", "odd_base", "padded"])
def test_leading_dims_and_offsets(config, layout):
    M, N, K = 133, 66, 35
    A, B, C0 = gen(M, N, K, seed=7)
    C, guards, plan = gpu_util.run(1.1, A, B, 0.5, C0, **layout)
    assert guards, "wrote outside C (padding or guard band)"
    check_full(1.1, A, B, 0.5, C0, C)


def test_tma_chosen_only_when_aligned():
    # 128 x 128: operands that TMA cannot describe are read too rarely to be
    # worth an aligned copy, so they take cp.async.
    A, B, C0 = gen(128, 128, 256, seed=8)
    _, _, plan = gpu_util.run(1.0, A, B, 0.0, C0)
    # Both by TMA in place (A row-major, "Atma", or transposed in shared
    # memory, "Axp"), no packing copy.
    assert ("Axp_Btma" in plan[0] or "Atma_Btma" in plan[0]) and "pack" not in plan[0], plan
    _, _, plan = gpu_util.run(1.0, A, B, 0.0, C0, lda=257)
    assert "Acp_Btma" in plan[0], plan
    _, _, plan = gpu_util.run(1.0, A, B, 0.0, C0, offsets=(0, 1, 0))
    assert "Atma_Bcp" in plan[0], plan


@pytest.mark.parametrize("layout,tags", [
    (dict(lda=1003), ["+packA"]),
    (dict(ldb=515), ["+packB"]),
    (dict(lda=1001, ldb=514, offsets=(1, 3, 0)), ["+packA", "+packB"]),
    (dict(offsets=(2, 0, 1), ldc=513), ["+packA"]),
], ids=["A", "B", "AB", "A_base_C_odd"])
def test_unaligned_operands_packed_then_tma(layout, tags):
    M, N, K = 300, 512, 1000
    A, B, C0 = gen(M, N, K, seed=9)
    C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0, **layout)
    assert guards
    assert "Atma_Btma" in plan[0] or "Axp_Btma" in plan[0], plan
    for t in tags:
        assert t in plan[0], plan
    check_full(0.7, A, B, -1.3, C0, C)
    # Forcing cp.async turns the copies off.
    assert sg.sgemm_set_config("auto:cpasync") == 0
    try:
        C2, _, plan2 = gpu_util.run(0.7, A, B, -1.3, C0, **layout)
        assert "pack" not in plan2[0] and "Acp_Bcp" in plan2[0], plan2
        check_full(0.7, A, B, -1.3, C0, C2)
    finally:
        sg.sgemm_set_config("auto")


@pytest.mark.parametrize("config", ["auto", "128x128", "64x64", "128x128:cpasync"], indirect=True)
def test_integer_inputs_bit_exact(config):
    w = inputs.WORKLOADS["sq1024_int"]
    A, B, C0 = w.make()
    C, guards, _ = gpu_util.run(w.alpha, A, B, w.beta, C0)
    assert guards
    check_full(w.alpha, A, B, w.beta, C0, C, exact=True)


def test_all_ones_closed_form():
    M, N, K = 300, 260, 777
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    C0 = inputs.fill("int", 9, inputs.TID_C, M, N)
    C, _, _ = gpu_util.run(2.0, A, B, -1.0, C0)
    assert np.array_equal(C, (2.0 * K - C0).astype(np.float32))


def test_identity_closed_form():
    n, N = 200, 150
    A = np.eye(n, dtype=np.float32)
    B = inputs.fill("normal", 10, inputs.TID_B, n, N)
    C, _, _ = gpu_util.run(1.0, A, B, 0.0, None)
    assert np.array_equal(C, B)


# ---- degenerate cases (BLAS readings) --------------------------------------

def test_beta_zero_never_reads_c():
    A, B, _ = gen(70, 90, 40, seed=11)
    C, _, _ = gpu_util.run(1.0, A, B, 0.0, None)          # C starts as NaN
    assert np.all(np.isfinite(C))
    check_full(1.0, A, B, 0.0, None, C)


def test_alpha_zero_scales_c_without_reading_ab():
    _, _, C0 = gen(50, 40, 30, seed=12)
    A = np.full((50, 30), np.nan, np.float32)
    B = np.full((30, 40), np.nan, np.float32)
    C, guards, plan = gpu_util.run(0.0, A, B, -1.5, C0)
    assert plan[0] == "scale" and guards
    assert np.array_equal(C, (np.float32(-1.5) * C0).astype(np.float32))
    C, _, _ = gpu_util.run(0.0, A, B, 0.0, None)
    assert np.array_equal(C, np.zeros_like(C))


def test_k_zero():
    _, _, C0 = gen(33, 17, 1, seed=13)
    A = np.zeros((33, 0), np.float32)
    B = np.zeros((0, 17), np.float32)
    C, guards, plan = gpu_util.run(2.0, A, B, 0.25, C0)
    assert plan[0] == "scale" and guards
    assert np.array_equal(C, (np.float32(0.25) * C0).astype(np.float32))


def test_empty_m_or_n_leaves_c_alone():
    torch = pytest.importorskip("torch")
    A, B, C0 = gen(4, 4, 4, seed=14)
    for (M, N) in [(0, 4), (4, 0)]:
        dA = torch.zeros(M, 4, device="cuda")
        dB = torch.zeros(4, N, device="cuda")
        dC = torch.zeros(M, N, device="cuda")
        sg.sgemm_tensors(1.0, dA, dB, 0.0, dC)
    torch.cuda.synchronize()


# ---- streams, repeat calls, status word -------------------------------------

def test_runs_on_a_side_stream_in_order():
    torch = pytest.importorskip("torch")
    M = N = K = 512
    A, B, C0 = gen(M, N, K, seed=15)
    s = torch.cuda.Stream()
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        dC = torch.from_numpy(C0).to("cuda", non_blocking=False)
        for _ in range(3):                     # C = 0.5 AB + 1 C, three times in order
            sg.sgemm_tensors(0.5, dA, dB, 1.0, dC, stream=s)
    s.synchronize()
    ref, S = oracle.sgemm_ref(1.5, A, B, 1.0, C0)
    rep = oracle.check(dC.cpu().numpy(), ref, 3 * S, K * 3)
    assert rep["ok"], rep


def test_bounded_wait_times_out_and_context_survives():
    torch = pytest.importorskip("torch")
    assert sg.check_status() == 0
    assert sg.sgemm_selftest_wait_timeout(20_000_000) == 0       # 20 ms
    rc, bits = sg.sgemm_check_status(torch.cuda.current_stream().cuda_stream)
    assert rc == sg.SGEMM_ERR_DEVICE_TIMEOUT and bits == 1
    assert sg.check_status() == 0                                 # cleared
    A, B, C0 = gen(64, 64, 64, seed=16)
    C, _, _ = gpu_util.run(1.0, A, B, 1.0, C0)                    # still usable
    check_full(1.0, A, B, 1.0, C0, C)


def test_fp32_peak_is_plausible():
    torch = pytest.importorskip("torch")
    props = torch.cuda.get_device_properties(0)
    datasheet = props.multi_processor_count * 128 * 2 * 2.07  # GFLOP/s at 2070 MHz
    got = {}
    for form in (sg.SGEMM_PEAK_FFMA, sg.SGEMM_PEAK_FFMA2, sg.SGEMM_PEAK_OUTER):
        r = sg.fp32_peak(target_ms=50, form=form)
        assert 0.2 * datasheet < r["gflops"] < 1.05 * datasheet, (form, r, datasheet)
        assert r["ms"] > 10
        got[form] = r["gflops"]
    # The outer product's 32 packed FMAs per k-step cannot outrun independent
    # packed-FMA chains.
    assert got[sg.SGEMM_PEAK_OUTER] < 1.02 * got[sg.SGEMM_PEAK_FFMA2], got


# ---- the five workloads, in the launch configuration the bench times --------

def _workload(name, full):
    torch = pytest.importorskip("torch")
    w = inputs.WORKLOADS[name]
    A, B, C0 = w.make()
    C, guards, plan = gpu_util.run(w.alpha, A, B, w.beta, C0 if w.beta != 0 else None)
    assert guards
    c0 = C0 if w.beta != 0 else None
    if full:
        rep = check_full(w.alpha, A, B, w.beta, c0, C, exact=w.exact)
    else:
        rows, cols = inputs.sample_entries(w.M, w.N)
        ref, S = oracle.sgemm_ref_sampled(w.alpha, A, B, w.beta, c0, rows, cols)
        rep = oracle.check(C[rows, cols], ref, S, w.K, exact=w.exact)
        assert rep["ok"], rep
    assert np.all(np.isfinite(C))
    return rep, plan


def test_workload_sq256_uniform():
    rep, plan = _workload("sq256_uniform", full=True)
    # A tile per 4-CTA cluster, 2 k-iterations each: A read row-major in place.
    assert plan[0] == "ws_64x64x32_s4_k4_c4_Atma_Btma", plan


def test_workload_sq1024_int_bit_exact():
    _workload("sq1024_int", full=True)


def test_workload_sq4096_uniform_sampled():
    rep, plan = _workload("sq4096_uniform", full=False)
    assert "128x128" in plan[0]


def test_workload_ragged_every_element():
    rep, plan = _workload("ragged_4093x5120x1531_normal", full=True)
    # A (6.3 M floats, lda = 1531) is copied transposed into an aligned
    # buffer and read through the transposed-A path.
    assert "ATtma_Btma+packAT" in plan[0], plan


def test_workload_llm_projection_sampled():
    _workload("llm_8192x14336x4096", full=False)


# ---- every compiled kernel family (tuning alternatives included) ------------

def _family_names():
    rc, names = sg.sgemm_config_names()
    assert rc == 0 and names
    return names


@pytest.mark.parametrize("cp", ["", ":cpasync"])
def test_every_family_matches_oracle(cp):
    for name in _family_names():
        assert sg.sgemm_set_config(name + cp) == 0, name
        try:
            for (M, N, K) in [(129, 257, 95), (256, 128, 64), (7, 300, 33)]:
                A, B, C0 = gen(M, N, K, seed=M + N + K)
                C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
                assert guards, (name, plan)
                assert plan[0].startswith(name), (name, plan)
                check_full(0.7, A, B, -1.3, C0, C)
        finally:
            sg.sgemm_set_config("auto")


def _ksplit(name):
    # Families whose warps split each stage's k into groups ("_k2", "_k4"),
    # also with their CTAs in clusters that split each tile's k ("_c2", "_c4").
    return re.search(r"_k[0-9]+(_c[0-9]+)?$", name) is not None


def test_families_agree_bitwise():
    # Under the data-parallel schedule every family accumulates each output
    # in the same k order with single-rounding FMAs, so they must agree bit
    # for bit (only the instruction schedule differs). The k-split families
    # add their groups' partial sums at the end instead, so they are held to
    # the bound (test_every_family_matches_oracle) and to determinism
    # (test_ksplit_families_are_deterministic) but not to these bits.
    torch = pytest.importorskip("torch")
    M, N, K = 640, 512, 768
    A, B, C0 = gen(M, N, K, seed=77)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    outs = {}
    for name in [n for n in _family_names() if not _ksplit(n)]:
        assert sg.sgemm_set_config(name + ":dp") == 0
        dC = torch.from_numpy(C0).cuda()
        sg.sgemm_tensors(0.7, dA, dB, -1.3, dC)
        sg.check_status()
        outs[name] = dC.cpu().numpy()
    sg.sgemm_set_config("auto")
    names = list(outs)
    for n in names[1:]:
        assert np.array_equal(outs[names[0]], outs[n]), (names[0], n)


def test_ksplit_families_are_deterministic():
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 700, 1300
    A, B, C0 = gen(M, N, K, seed=78)
    for name in [n for n in _family_names() if _ksplit(n)]:
        outs = []
        for cfg in (name, name, name + ":dp"):
            assert sg.sgemm_set_config(cfg) == 0
            try:
                C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
            finally:
                sg.sgemm_set_config("auto")
            assert guards and plan[0].startswith(name), (cfg, plan)
            outs.append(C)
        assert np.array_equal(outs[0], outs[1]), name
        for C in (outs[0], outs[2]):
            check_full(0.7, A, B, -1.3, C0, C)


# ---- the stream-K tail ----------------------------------------------------------

SK_SHAPES = [
    (1024, 1024, 1024),     # 64 tiles < 152 SMs: every tile split
    (256, 512, 2048),       # 8 tiles of 64 k-tiles over 152 CTAs: ~19 parts per tile
    (128, 128, 16384),      # one tile, 512 k-tiles: 32 parts
    (512, 5504, 96),        # 172 tiles: one full wave + a 20-tile tail
    (333, 4500, 777),       # ragged edges, 1 wave + tail
    (130, 70, 8400),        # tiles cut by both edges, 29 parts per tile
]


@pytest.mark.parametrize("cp", ["", ":cpasync"])
@pytest.mark.parametrize("shape", SK_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stream_k_tail_matches_oracle(shape, cp):
    # The 128 x 128 family forced: its fixed rule splits every partial last
    # wave below 90 % of the SMs (auto may prefer the 128 x 64 tile here).
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=200 + M % 97 + N % 89 + K % 83)
    assert sg.sgemm_set_config("128x128" + cp) == 0
    try:
        C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
        assert guards
        assert plan[0].endswith("+sk"), plan
        check_full(0.7, A, B, -1.3, C0, C)
        # beta == 0 through the fixup: C is not read.
        C, guards, plan = gpu_util.run(1.5, A, B, 0.0, None)
        assert guards and plan[0].endswith("+sk"), plan
        check_full(1.5, A, B, 0.0, None, C)
    finally:
        sg.sgemm_set_config("auto")


def test_stream_k_is_deterministic_and_close_to_dp():
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 1100, 2000
    A, B, C0 = gen(M, N, K, seed=300)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    outs = []
    # The 128 x 128 family forced: its 72 tiles leave SMs idle, so every tile
    # is split ("auto" takes the 128 x 64 k-group tile here instead).
    try:
        for cfg in ["128x128", "128x128", "128x128:dp"]:
            assert sg.sgemm_set_config(cfg) == 0
            dC = torch.from_numpy(C0).cuda()
            name, _ = sg.plan_tensors(0.7, dA, dB, -1.3, dC)
            assert name.endswith("+sk") == (cfg == "128x128"), name
            sg.sgemm_tensors(0.7, dA, dB, -1.3, dC)
            sg.check_status()
            outs.append(dC.cpu().numpy())
    finally:
        sg.sgemm_set_config("auto")
    assert np.array_equal(outs[0], outs[1])          # same schedule, same bits
    for C in (outs[0], outs[2]):
        check_full(0.7, A, B, -1.3, C0, C)


def test_integer_inputs_bit_exact_with_stream_k():
    A = inputs.fill("int", 5, inputs.TID_A, 700, 1500)
    B = inputs.fill("int", 5, inputs.TID_B, 1500, 900)
    C0 = inputs.fill("int", 5, inputs.TID_C, 700, 900)
    assert sg.sgemm_set_config("128x128") == 0
    try:
        C, _, plan = gpu_util.run(2.0, A, B, -1.0, C0)
    finally:
        sg.sgemm_set_config("auto")
    assert plan[0].endswith("+sk"), plan
    check_full(2.0, A, B, -1.0, C0, C, exact=True)


@pytest.mark.parametrize("cfg", ["ws_64x64x32_s4_k4", "ws_64x64x32_s4_k4:cpasync:dp",
                                 "ws_128x64x32_s4_k2:dp", "ws_64x64x32_s4_k2"])
def test_integer_inputs_bit_exact_on_ksplit_tiles(cfg):
    # The k-groups' partial sums are integers below 2^24 here, so adding
    # them at the end changes no bit.
    A = inputs.fill("int", 6, inputs.TID_A, 333, 1500)
    B = inputs.fill("int", 6, inputs.TID_B, 1500, 517)
    C0 = inputs.fill("int", 6, inputs.TID_C, 333, 517)
    assert sg.sgemm_set_config(cfg) == 0
    try:
        C, guards, plan = gpu_util.run(2.0, A, B, -1.0, C0)
    finally:
        sg.sgemm_set_config("auto")
    assert guards and plan[0].startswith(cfg.split(":")[0]), plan
    check_full(2.0, A, B, -1.0, C0, C, exact=True)


@pytest.mark.parametrize("cfg", ["ws_64x64x32_s4_k4_c2", "ws_64x64x32_s4_k4_c4",
                                 "ws_64x64x32_s4_k4_c4:cpasync", "ws_64x64x32_s4_k4_c4:at"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 7, 33), (64, 64, 96), (256, 256, 256),
                                   (300, 512, 1000), (1000, 700, 1300), (130, 72, 4100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_cluster_k_split_matches_oracle(cfg, shape):
    # The CTAs of a cluster share a tile, each a share of its k-tiles (none
    # at all when K has fewer k-tiles than the cluster has CTAs), and the
    # first adds the others' sums, read from its shared memory.
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=95)
    assert sg.sgemm_set_config(cfg) == 0
    try:
        C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
        C1, guards1, _ = gpu_util.run(1.5, A, B, 0.0, None)
    finally:
        sg.sgemm_set_config("auto")
    assert guards and guards1 and plan[0].startswith(cfg.split(":")[0] + "_"), plan
    assert "+sk" not in plan[0], plan
    check_full(0.7, A, B, -1.3, C0, C)
    check_full(1.5, A, B, 0.0, None, C1)


def test_cluster_k_split_integers_bit_exact_and_deterministic():
    A = inputs.fill("int", 7, inputs.TID_A, 300, 2000)
    B = inputs.fill("int", 7, inputs.TID_B, 2000, 200)
    C0 = inputs.fill("int", 7, inputs.TID_C, 300, 200)
    outs = []
    for cfg in ["ws_64x64x32_s4_k4_c4", "ws_64x64x32_s4_k4_c4", "ws_64x64x32_s4_k4_c2"]:
        assert sg.sgemm_set_config(cfg) == 0
        try:
            C, guards, plan = gpu_util.run(2.0, A, B, -1.0, C0)
        finally:
            sg.sgemm_set_config("auto")
        assert guards, plan
        check_full(2.0, A, B, -1.0, C0, C, exact=True)
        outs.append(C)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("shape", [(256, 256, 8192), (200, 300, 6000), (130, 72, 4100)],
                         ids=lambda s: "x".join(map(str, s)))
def test_auto_splits_deep_k_over_small_tiles(shape):
    # Few tiles and a deep K: "auto" takes the 64 x 64 tile in four k-groups
    # and spreads its k-iterations over the SMs (stream-K tail).
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=91)
    C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
    assert guards and plan[0].startswith("ws_64x64x32_s4_k4_") and plan[0].endswith("+sk"), plan
    check_full(0.7, A, B, -1.3, C0, C)


# ---- streams and graphs ----------------------------------------------------------

def test_two_streams_concurrently_do_not_share_workspace():
    # Both problems take the stream-K tail (a per-call workspace); run them
    # back to back on two streams with no ordering between them.
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 1100, 2000
    A1, B1, C1 = gen(M, N, K, seed=401)
    A2, B2, C2 = gen(M, N, K, seed=402)
    d = [torch.from_numpy(x).cuda() for x in (A1, B1, C1, A2, B2, C2)]
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
    check_full(0.7, A1, B1, -1.3, C1, c1.cpu().numpy())
    check_full(0.7, A2, B2, -1.3, C2, c2.cpu().numpy())


def test_host_threads_call_concurrently():
    # Four host threads, each on its own stream, plan and launch at the same
    # time (ctypes drops the GIL during the call): the library's per-device
    # set-up, shape rules and workspace pool are shared between them.
    import threading
    torch = pytest.importorskip("torch")
    shapes = [(1000, 1100, 2000), (700, 900, 1500), (333, 4500, 776), (2048, 2048, 1024)]
    cases = [gen(M, N, K, seed=410 + i) for i, (M, N, K) in enumerate(shapes)]
    dev = [(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), torch.from_numpy(C0).cuda())
           for A, B, C0 in cases]
    c0s = [torch.from_numpy(C0).cuda() for _, _, C0 in cases]
    streams = [torch.cuda.Stream() for _ in shapes]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(len(shapes))

    def work(i):
        try:
            dA, dB, dC = dev[i]
            start.wait()
            for _ in range(3):
                with torch.cuda.stream(streams[i]):
                    dC.copy_(c0s[i])
                    sg.sgemm_tensors(0.7, dA, dB, -1.3, dC, stream=streams[i])
                streams[i].synchronize()
        except Exception as e:          # reported below, on the main thread
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(shapes))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    sg.check_status()
    for (A, B, C0), (_, _, dC) in zip(cases, dev):
        check_full(0.7, A, B, -1.3, C0, dC.cpu().numpy())


def test_sgemm_inside_a_captured_cuda_graph():
    # The stream-K workspace is stream-ordered, so capture records it as an
    # allocation node; the graph replays correctly. (The first call on the
    # device, which allocates the status word, happens before capture.)
    torch = pytest.importorskip("torch")
    M, N, K = 1000, 1100, 2000
    A, B, C0 = gen(M, N, K, seed=403)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    assert sg.sgemm_set_config("128x128") == 0      # 72 tiles: every one split
    try:
        name, _ = sg.plan_tensors(0.7, dA, dB, -1.3, dC)
        assert name.endswith("+sk"), name
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            sg.sgemm_tensors(0.7, dA, dB, -1.3, dC.clone(), stream=s)   # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        work = dC.clone()
        with torch.cuda.graph(g):
            sg.sgemm_tensors(0.7, dA, dB, -1.3, work)
        for _ in range(2):
            work.copy_(dC)
            g.replay()
        torch.cuda.synchronize()
        sg.check_status()
    finally:
        sg.sgemm_set_config("auto")
    check_full(0.7, A, B, -1.3, C0, work.cpu().numpy())


def test_copy_then_gemm_inside_a_captured_cuda_graph():
    # 2048 x 2048 x 4096 takes the transposed copy of A, and the GEMM behind
    # it is launched by programmatic stream serialisation: capture records
    # that as a programmatic edge, and replays give the oracle's result.
    torch = pytest.importorskip("torch")
    M, N, K = 2048, 2048, 4096
    A, B, C0 = gen(M, N, K, seed=404)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C0).cuda()
    name, _ = sg.plan_tensors(0.7, dA, dB, -1.3, dC)
    assert "+packAT" in name, name
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sg.sgemm_tensors(0.7, dA, dB, -1.3, dC.clone(), stream=s)       # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    work = dC.clone()
    with torch.cuda.graph(g):
        sg.sgemm_tensors(0.7, dA, dB, -1.3, work)
    for _ in range(3):
        work.copy_(dC)
        g.replay()
    torch.cuda.synchronize()
    sg.check_status()
    C = work.cpu().numpy()
    rows, cols = inputs.sample_entries(M, N)
    ref, S = oracle.sgemm_ref_sampled(0.7, A, B, -1.3, C0, rows, cols)
    rep = oracle.check(C[rows, cols], ref, S, K)
    assert rep["ok"], rep
    # Eager calls give the same bits as the replays.
    eager = dC.clone()
    sg.sgemm_tensors(0.7, dA, dB, -1.3, eager)
    sg.check_status()
    assert np.array_equal(eager.cpu().numpy(), C)


def test_programmatic_launch_changes_no_bit():
    # The same 2048 x 2048 x 4096 call in a process with SGEMM_PDL=0 (every
    # kernel launched the ordinary way) gives the same bits.
    import os
    import subprocess
    import sys
    torch = pytest.importorskip("torch")
    M, N, K = 2048, 2048, 4096
    A, B, C0 = gen(M, N, K, seed=405)
    dC = torch.from_numpy(C0).cuda()
    sg.sgemm_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)
    sg.check_status()
    here = dC.cpu().numpy()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = (
        "import sys, numpy as np, torch\n"
        "import dense_fp32_matrix_strict_gb300 as sg\n"
        "from dense_fp32_matrix_strict_gb300 import inputs as I\n"
        f"A = I.fill('normal', 405, I.TID_A, {M}, {K})\n"
        f"B = I.fill('normal', 405, I.TID_B, {K}, {N})\n"
        f"C0 = I.fill('normal', 405, I.TID_C, {M}, {N})\n"
        "dC = torch.from_numpy(C0).cuda()\n"
        "sg.sgemm_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)\n"
        "sg.check_status()\n"
        "sys.stdout.buffer.write(dC.cpu().numpy().tobytes())\n")
    env = dict(os.environ, SGEMM_PDL="0")
    out = subprocess.run([sys.executable, "-c", script], cwd=root, env=env, capture_output=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr.decode()[-2000:]
    there = np.frombuffer(out.stdout, dtype=np.float32).reshape(M, N)
    assert np.array_equal(here, there)


@pytest.mark.parametrize("shape", [(2304, 2304, 1024), (512, 640, 500)],
                         ids=["cta_pairs_256", "tiles_128"])
def test_programmatic_launch_changes_no_bit_3xtf32(shape):
    # sgemm_3xtf32 runs its B split alongside the A split and the MMA kernel
    # behind them by programmatic stream serialisation; with SGEMM_PDL=0
    # (ordinary launches) the bits are the same. 2304^2 takes the CTA-pair
    # kernel (81 tiles of 256 x 256), 512 x 640 the 128 x 128 kernel.
    import os
    import subprocess
    import sys
    torch = pytest.importorskip("torch")
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=406)
    dC = torch.from_numpy(C0).cuda()
    sg.sgemm_3xtf32_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)
    sg.check_status()
    here = dC.cpu().numpy()
    ref, S = oracle.sgemm_ref(0.7, A, B, -1.3, C0)
    assert oracle.check(here, ref, S, K)["ok"]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = (
        "import sys, numpy as np, torch\n"
        "import dense_fp32_matrix_strict_gb300 as sg\n"
        "from dense_fp32_matrix_strict_gb300 import inputs as I\n"
        f"A = I.fill('normal', 406, I.TID_A, {M}, {K})\n"
        f"B = I.fill('normal', 406, I.TID_B, {K}, {N})\n"
        f"C0 = I.fill('normal', 406, I.TID_C, {M}, {N})\n"
        "dC = torch.from_numpy(C0).cuda()\n"
        "sg.sgemm_3xtf32_tensors(0.7, torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), -1.3, dC)\n"
        "sg.check_status()\n"
        "sys.stdout.buffer.write(dC.cpu().numpy().tobytes())\n")
    env = dict(os.environ, SGEMM_PDL="0")
    out = subprocess.run([sys.executable, "-c", script], cwd=root, env=env, capture_output=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr.decode()[-2000:]
    there = np.frombuffer(out.stdout, dtype=np.float32).reshape(M, N)
    assert np.array_equal(here, there)


@pytest.mark.parametrize("config", ["128x128", "128x128:dp", "128x64:dp", "64x64:dp"])
@pytest.mark.parametrize("aligned", [True, False], ids=["aligned", "unaligned"])
def test_a_paths_give_the_same_bits(config, aligned):
    # How a row-major A reaches the consumers -- as stored (":noat"), through
    # a transposed copy in HBM (":at") or transposed in shared memory by the
    # kernel (":xp", aligned A only) -- changes no output bit: every output
    # sees the same FMA sequence. (With the stream-K tail that holds only at
    # equal grids: the split follows the CTAs per SM of the variant, which is
    # one for every 128 x 128 variant; the 64 x 64 variants differ, so that
    # family is compared under ":dp".)
    M, N, K = 700, 900, 1500
    A, B, C0 = gen(M, N, K, seed=61)
    layout = {} if aligned else dict(lda=K + 1, offsets=(1, 0, 0))
    outs, plans = [], []
    for mod in (":noat", ":at", ":xp"):
        assert sg.sgemm_set_config(config + mod) == 0
        try:
            C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0, **layout)
        finally:
            sg.sgemm_set_config("auto")
        assert guards
        outs.append(C)
        plans.append(plan[0])
    assert "+packAT" not in plans[0] and "ATtma" not in plans[0] and "Axp" not in plans[0], plans
    assert "_ATtma_" in plans[1] and "+packAT" in plans[1], plans
    if aligned:
        assert "_Axp_Btma" in plans[2], plans
    for C in outs[1:]:
        assert np.array_equal(outs[0], C), plans
    check_full(0.7, A, B, -1.3, C0, outs[2])


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (333, 4500, 776), (130, 72, 8400),
                                   (4093, 5120, 1536)], ids=lambda s: "x".join(map(str, s)))
def test_in_smem_transpose_with_stream_k(shape):
    # Leading dimensions K and N multiples of 4: both operands go by TMA in
    # place, the condition for the in-smem transpose.
    M, N, K = shape
    A, B, C0 = gen(M, N, K, seed=71)
    assert sg.sgemm_set_config("128x128:xp") == 0
    try:
        C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0)
    finally:
        sg.sgemm_set_config("auto")
    assert guards and "_Axp_Btma" in plan[0], plan
    check_full(0.7, A, B, -1.3, C0, C)


def test_auto_a_path_by_size():
    # Large: the transposed copy of A pays. Medium and small: the in-smem
    # transpose, unless a CTA's work item has under 4 k-iterations (256^3 in
    # clusters of 4), where A is read row-major in place. An A TMA cannot
    # read in place: the copy where it pays.
    torch = pytest.importorskip("torch")
    def plan(M, N, K, lda=None):
        A = torch.empty(M, lda or K, device="cuda")[:, :K]
        B = torch.empty(K, N, device="cuda")
        C = torch.empty(M, N, device="cuda")
        return sg.plan_tensors(1.0, A, B, 0.0, C)[0]
    assert "_ATtma_Btma+packAT" in plan(4096, 4096, 4096)
    assert "_Axp_Btma" in plan(2048, 2048, 2048)
    assert "_Atma_Btma" in plan(256, 256, 256)
    assert "_Axp_Btma" in plan(640, 640, 640)
    assert "_ATtma_Btma+packAT" in plan(2048, 2048, 2047, lda=2047)
