"""When a call takes the transposed copy of A ("+packAT"): the size rule.

sgemm reads a row-major A through the k-major ([k][m]) shared-memory layout,
which keeps the FFMA pipe busier than the row-major read. It gets there
either by transposer warps inside the kernel (no workspace) or by a
transposed copy of A in a stream-ordered workspace first (one HBM read and
write of A, plus a launch). The copy is taken when its extra saving on the
main loop pays for it:

    t_main = 2 M N K / 66e12 s          (the main loop at ~66 TFLOP/s)
    cost   = 5e-6 + 8 M K / 6e12 s      (launch + pool, A read and written at ~6 TB/s)
    copy  <=>  f * t_main > cost,  f = 0.036 where the in-kernel transpose is
               available to the chosen family and a CTA's work item has at
               least 4 k-iterations, else 0.085.

The rule is written out here on its own, independently of the library; the
CPU test pins it on the five workloads, the GPU test checks sgemm_plan
against it over a grid of shapes.
"""
import pytest

import dense_fp32_matrix_strict_gb300 as sg


def cdiv(a, b):
    return (a + b - 1) // b


def takes_transposed_copy(M, N, K, xp_auto):
    t_main = 2.0 * M * N * K / 66e12
    cost = 5e-6 + 8.0 * M * K / 6e12
    return (0.036 if xp_auto else 0.085) * t_main > cost


def family_of(plan):
    """(tile family, CTAs per cluster) from a plan name such as
    "ws_64x64x32_s4_k4_c2_Axp_Btma"."""
    if plan.startswith("ws_128x64x32_s4_") and "_k2_" not in plan:
        fam = "128x64"
    else:
        fam = plan.split("_")[1]
    cs = 4 if "_c4_" in plan else 2 if "_c2_" in plan else 1
    return fam, cs


def test_rule_on_the_five_workloads():
    # 4096^3, the LLM projection and the ragged shape take the copy; the
    # two small ones do not. (The ragged A, lda = 1531, cannot be read by
    # TMA in place, so no in-kernel transpose: f = 0.085.)
    assert takes_transposed_copy(4096, 4096, 4096, True)
    assert takes_transposed_copy(8192, 14336, 4096, True)
    assert takes_transposed_copy(4093, 5120, 1531, False)
    assert not takes_transposed_copy(1024, 1024, 1024, True)
    assert not takes_transposed_copy(256, 256, 256, False)
    # Near the boundary: 2048^3 stays with the in-kernel transpose, 2048^2 x
    # 8192 takes the copy.
    assert not takes_transposed_copy(2048, 2048, 2048, True)
    assert takes_transposed_copy(2048, 2048, 8192, True)


SHAPES = [(m, n, k) for m in (512, 1024, 2048, 3072, 4096) for n in (1024, 2048, 4096)
          for k in (512, 2048, 8192)] + [(8192, 14336, 4096), (4096, 4096, 4096)]


@pytest.mark.gpu
def test_plan_takes_the_copy_exactly_where_the_rule_says():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    assert sg.sgemm_set_config("auto") == 0
    # Planning reads no memory: distinct, aligned placeholder addresses.
    A, B, C = 1 << 36, 2 << 36, 3 << 36
    seen = set()
    for (M, N, K) in SHAPES:
        rc, plan, _ = sg.sgemm_plan(M, N, K, 1.0, A, K, B, N, 0.0, C, N)
        assert rc == 0, (M, N, K, rc)
        fam, cs = family_of(plan)
        item_kt = cdiv(cdiv(K, 32), cs)
        # Every operand here is TMA-aligned, so the in-kernel transpose is
        # open to every family but the two-CTA 128 x 64 tile.
        xp_auto = fam != "128x64" and item_kt >= 4
        want = takes_transposed_copy(M, N, K, xp_auto)
        assert ("+packAT" in plan) == want, (M, N, K, plan)
        seen.add(want)
    assert seen == {True, False}
