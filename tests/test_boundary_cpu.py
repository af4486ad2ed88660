"""The C ABI on the CPU: the library loads, exports what include/sgemm.h
declares, and rejects bad arguments before touching a GPU."""
import os
import re

import pytest

import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sg.load()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                text = f.read()
            names += re.findall(r"^SGEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_binding_symbols():
    assert sorted(declared_functions()) == sorted(sg.EXPORTED_SYMBOLS)


def test_header_constants_match_the_binding():
    # Every SGEMM_* constant the header defines has the binding's value.
    with open(os.path.join(ROOT, "include", "sgemm.h")) as f:
        text = f.read()
    defs = dict(re.findall(r"^#define (SGEMM_(?:ERR|OK|OP|PEAK)\w*)\s+(\d+)", text, flags=re.M))
    assert {"SGEMM_OK", "SGEMM_PEAK_FFMA", "SGEMM_PEAK_FFMA2", "SGEMM_PEAK_OUTER"} <= set(defs)
    for name, value in defs.items():
        assert getattr(sg, name) == int(value), name


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_library_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", sg.library_path()],
                         capture_output=True, text=True, check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert syms == set(declared_functions())


def test_error_strings(lib):
    for code in range(7):
        assert sg.sgemm_error_string(code)
    assert sg.sgemm_error_string(99) == "unknown error code"


# (M, N, K, alpha, A, lda, B, ldb, beta, C, ldc) that violate the contract.
A_PTR, B_PTR, C_PTR = 1 << 20, 2 << 20, 3 << 20
BAD_ARGS = [
    (-1, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),            # negative M
    (4, -1, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),            # negative N
    (4, 4, -1, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),            # negative K
    (1 << 31, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),       # M too large
    (4, 4, 8, 1.0, A_PTR, 7, B_PTR, 4, 0.0, C_PTR, 4),             # lda < K
    (4, 8, 4, 1.0, A_PTR, 4, B_PTR, 7, 0.0, C_PTR, 8),             # ldb < N
    (4, 8, 4, 1.0, A_PTR, 4, B_PTR, 8, 0.0, C_PTR, 7),             # ldc < N
    (4, 4, 4, 1.0, 0, 4, B_PTR, 4, 0.0, C_PTR, 4),                 # A NULL
    (4, 4, 4, 1.0, A_PTR, 4, 0, 4, 0.0, C_PTR, 4),                 # B NULL
    (4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, 0, 4),                 # C NULL
    (4, 4, 4, 1.0, A_PTR + 2, 4, B_PTR, 4, 0.0, C_PTR, 4),         # A misaligned
    (4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR + 1, 4),         # C misaligned
    (4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, A_PTR + 32, 4),        # C overlaps A
    (4, 4, 4, 1.0, A_PTR, 4, C_PTR - 16, 4, 0.0, C_PTR, 4),        # C overlaps B
    (4, 4, 4, 1.0, A_PTR, 1 << 62, B_PTR, 4, 0.0, C_PTR, 4),       # lda overflows offsets
]


@pytest.mark.parametrize("args", BAD_ARGS)
def test_invalid_arguments_rejected_without_gpu(lib, args):
    assert sg.sgemm(*args, 0) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_plan(*args)[0] == sg.SGEMM_ERR_INVALID_VALUE


def test_empty_problem_is_a_no_op(lib):
    assert sg.sgemm(0, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4, 0) == sg.SGEMM_OK
    assert sg.sgemm(4, 0, 4, 1.0, A_PTR, 4, B_PTR, 1, 0.0, C_PTR, 1, 0) == sg.SGEMM_OK
    assert sg.sgemm_plan(0, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4) == (0, "none", 0)


def test_null_ab_allowed_when_not_read(lib):
    # alpha == 0 or K == 0: A and B are not read, so NULL passes the checks
    # (the call then needs a device; without one it reports a CUDA error).
    rc = sg.sgemm(4, 4, 4, 0.0, 0, 4, 0, 4, 1.0, C_PTR, 4, 0)
    assert rc != sg.SGEMM_ERR_INVALID_VALUE
    rc = sg.sgemm(4, 4, 0, 1.0, 0, 1, 0, 4, 1.0, C_PTR, 4, 0)
    assert rc != sg.SGEMM_ERR_INVALID_VALUE


def test_config_names(lib):
    for good in ["auto", "128x128", "64x64", "128x64", "128x128:cpasync", "auto:cpasync",
                 "auto:at", "128x128:noat:dp", "128x128:fixup", "auto:dp:fixup",
                 "auto:dp:atcopy"]:
        assert sg.sgemm_set_config(good) == sg.SGEMM_OK
    for bad in ["", "x", "256x256", "128x128:tma", "auto:"]:
        if bad == "":
            continue
        assert sg.sgemm_set_config(bad) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_set_config("auto") == sg.SGEMM_OK


def test_timeout_setting_bounds(lib):
    assert sg.sgemm_set_wait_timeout_ns(10) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_set_wait_timeout_ns(2_000_000_000) == sg.SGEMM_OK
    assert sg.sgemm_selftest_wait_timeout(10) == sg.SGEMM_ERR_INVALID_VALUE


def test_occupy_selftest_argument_checks(lib):
    for ctas, ns in [(0, 1000), (-1, 1000), (1, 0), (1, 2_000_000_001)]:
        assert sg.sgemm_selftest_occupy(ctas, ns) == sg.SGEMM_ERR_INVALID_VALUE
    # Valid arguments on a machine without a GPU: an error, never SGEMM_OK.
    assert sg.sgemm_selftest_occupy(1, 1000) != sg.SGEMM_OK


def test_tensor_wrapper_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    a = torch.zeros(4, 4)
    with pytest.raises(TypeError):
        sg.sgemm_tensors(1.0, a, a, 0.0, a.clone())


def test_shape_config_rules(lib):
    assert sg.sgemm_set_shape_config(-1, 4, 4, "128x128") == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_set_shape_config(4, 4, 4, "256x256") == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_set_shape_config(4, 4, 4, "64x64:dp") == sg.SGEMM_OK
    assert sg.sgemm_set_shape_config(4, 4, 4, "128x128") == sg.SGEMM_OK   # replaces
    assert sg.sgemm_set_shape_config(4, 4, 4, "auto") == sg.SGEMM_OK      # removes
    assert sg.sgemm_set_shape_config(4, 4, 4, None) == sg.SGEMM_OK        # absent: no-op
    # The table holds 256 shapes; a 257th new shape is refused, an update is not.
    for i in range(256):
        assert sg.sgemm_set_shape_config(1, 1, i + 1, "64x64") == sg.SGEMM_OK
    assert sg.sgemm_set_shape_config(1, 1, 1000, "64x64") == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_set_shape_config(1, 1, 7, "128x128") == sg.SGEMM_OK
    assert sg.sgemm_set_shape_config(1, 1, 7, "auto") == sg.SGEMM_OK
    assert sg.sgemm_set_shape_config(1, 1, 1000, "64x64") == sg.SGEMM_OK
    assert sg.sgemm_clear_shape_configs() == sg.SGEMM_OK


BAD_EX_ARGS = [
    (2, 0, 4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),          # opa not 0/1
    (0, -1, 4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4),         # opb not 0/1
    (1, 0, 8, 4, 4, 1.0, A_PTR, 7, B_PTR, 4, 0.0, C_PTR, 4),          # A^T: lda < M
    (0, 1, 4, 4, 8, 1.0, A_PTR, 8, B_PTR, 7, 0.0, C_PTR, 4),          # B^T: ldb < K
    (1, 1, 4, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, A_PTR + 32, 4),     # C overlaps A
    (1, 0, 4, 4, 4, 1.0, A_PTR, 1 << 62, B_PTR, 4, 0.0, C_PTR, 4),    # lda overflows (K rows)
]


@pytest.mark.parametrize("args", BAD_EX_ARGS)
def test_invalid_transposed_arguments_rejected_without_gpu(lib, args):
    assert sg.sgemm_ex(*args, 0) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_3xtf32_ex(*args, 0) == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_plan_ex(*args)[0] == sg.SGEMM_ERR_INVALID_VALUE


def test_transposed_leading_dimensions_follow_the_stored_shape(lib):
    # M = 8, K = 4: A^T is stored 4 x 8, so lda = 8 is the minimum; a plain
    # A (8 x 4) would accept lda = 4, the transposed one must not.
    assert sg.sgemm_plan_ex(1, 0, 8, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4)[0] == \
        sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_plan_ex(0, 0, 8, 4, 4, 1.0, A_PTR, 4, B_PTR, 4, 0.0, C_PTR, 4)[0] != \
        sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_ex(1, 1, 0, 4, 4, 1.0, A_PTR, 1, B_PTR, 4, 0.0, C_PTR, 4, 0) == sg.SGEMM_OK


def test_ceiling_forms_and_noalloc_status_without_gpu(lib):
    # An unknown instruction form or a bad target is refused before any
    # device work; the valid forms need a device and report a CUDA error here.
    assert sg.sgemm_fp32_peak_ex(3, 10.0)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_fp32_peak_ex(-1, 10.0)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_fp32_peak_ex(sg.SGEMM_PEAK_FFMA2, 0.5)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_fp32_peak_ex(sg.SGEMM_PEAK_OUTER, 0.5)[0] == sg.SGEMM_ERR_INVALID_VALUE
    for form in (sg.SGEMM_PEAK_FFMA, sg.SGEMM_PEAK_FFMA2, sg.SGEMM_PEAK_OUTER):
        rc = sg.sgemm_fp32_peak_ex(form, 10.0)[0]
        assert rc not in (sg.SGEMM_OK, sg.SGEMM_ERR_INVALID_VALUE)
    # The scratch status check needs the device's scratch address: without a
    # device it returns an error (never SGEMM_OK) and leaves `bits` alone;
    # a NULL `bits` is accepted.
    rc, bits = sg.sgemm_noalloc_check_status(0)
    assert rc not in (sg.SGEMM_OK, sg.SGEMM_ERR_DEVICE_TIMEOUT) and bits == 0
    assert sg.load().sgemm_noalloc_check_status(None, None) not in (
        sg.SGEMM_OK, sg.SGEMM_ERR_DEVICE_TIMEOUT)


def test_null_launch_without_gpu_is_a_launch_error(lib):
    assert sg.sgemm_null_launch(0) == sg.SGEMM_ERR_LAUNCH


def test_tf32_mma_peak_arguments(lib):
    assert sg.sgemm_tf32_mma_peak(64, 10.0)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_tf32_mma_peak(128, 0.0)[0] == sg.SGEMM_ERR_INVALID_VALUE
    assert sg.sgemm_tf32_mma_peak(256, 10.0)[0] not in (sg.SGEMM_OK, sg.SGEMM_ERR_INVALID_VALUE)
