"""An SGEMM started while another kernel holds half of the SMs.

The persistent GEMM kernel launches as many CTAs as the GPU runs at once.
With half of the SMs held by a kernel on another stream
(sgemm_selftest_occupy), only about half of them start; the others start as
SMs free up. Under the default plan some CTAs wait for others (the stream-K
tail's finishing CTA for the partial sums of higher-index CTAs, the TMA
producers for blocks of a copy made inside the kernel that any CTA may
write), so the call may wait for the other kernel to end; every wait is
bounded, and with the other kernel shorter than the wait limit the call must
come back with a clear status word and the bits of the same call on an idle
GPU. Under "auto:dp:atcopy" no CTA waits for another, so the call finishes
long before the other kernel does.
"""
import time

import numpy as np
import pytest

import dense_fp32_matrix_strict_gb300 as sg
from dense_fp32_matrix_strict_gb300 import inputs

pytestmark = pytest.mark.gpu

HOLD_NS = 400_000_000      # the other kernel holds its SMs for 0.4 s


@pytest.fixture(scope="module", autouse=True)
def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.load()
    sg.sgemm_set_config("auto")
    yield
    sg.sgemm_set_config("auto")


def _run_beside_holder(cfg, M, N, K, ta, tb, tags):
    """(C on an idle GPU, C while half the SMs are held, ms of the second
    call, whether the holder was still running when it ended)."""
    import torch
    A = inputs.fill("uniform", 91, inputs.TID_A, *((K, M) if ta else (M, K)))
    B = inputs.fill("uniform", 91, inputs.TID_B, *((N, K) if tb else (K, N)))
    C0 = inputs.fill("uniform", 91, inputs.TID_C, M, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    assert sg.sgemm_set_config(cfg) == 0
    try:
        name, _ = sg.plan_tensors(0.5, dA, dB, -1.0, torch.empty(M, N, device="cuda"),
                                  transa=ta, transb=tb)
        for tag in tags:
            assert tag in name, name
        dC = torch.from_numpy(C0).cuda()
        sg.sgemm_tensors(0.5, dA, dB, -1.0, dC, transa=ta, transb=tb)
        torch.cuda.synchronize()
        sg.check_status()
        want = dC.cpu().numpy()

        sms = torch.cuda.get_device_properties(0).multi_processor_count
        hold = torch.cuda.Stream()
        work = torch.cuda.Stream()
        dC2 = torch.from_numpy(C0).cuda()
        torch.cuda.synchronize()
        assert sg.sgemm_selftest_occupy(sms // 2, HOLD_NS, hold.cuda_stream) == 0
        time.sleep(0.05)                    # its CTAs are on their SMs by now
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(work):
            e0.record(work)
            sg.sgemm_tensors(0.5, dA, dB, -1.0, dC2, stream=work, transa=ta, transb=tb)
            e1.record(work)
        e1.synchronize()
        held = not hold.query()
        ms = e0.elapsed_time(e1)
        torch.cuda.synchronize()
        sg.check_status()                   # raises on a time-out
        return want, dC2.cpu().numpy(), ms, held
    finally:
        sg.sgemm_set_config("auto")


# (M, N, K, transa, transb, plan tags that must appear)
DEFAULT_CASES = [
    (4096, 4096, 4096, False, False, ("+packATfused", "+sk")),
    (4096, 4096, 4096, False, True, ("+packATfused", "+packBTfused", "+sk")),
    (2048, 2048, 2048, False, False, ("+sk",)),
]


@pytest.mark.parametrize("M,N,K,ta,tb,tags", DEFAULT_CASES,
                         ids=["x".join(map(str, c[:3])) + ("_T" if c[3] else "_N") +
                              ("T" if c[4] else "N") for c in DEFAULT_CASES])
def test_default_plan_is_correct_beside_a_kernel_holding_half_the_sms(M, N, K, ta, tb, tags):
    want, got, ms, _ = _run_beside_holder("auto", M, N, K, ta, tb, tags)
    assert ms < 2000.0, ms                  # within the wait limit, no time-out
    assert np.array_equal(got, want), int(np.count_nonzero(got != want))


def test_configuration_without_waits_finishes_while_half_the_sms_are_held():
    want, got, ms, held = _run_beside_holder("auto:dp:atcopy", 4096, 4096, 4096, False, False,
                                             ("+packAT",))
    assert held                             # the other kernel was still running
    assert ms < 150.0, ms                   # did not wait for its 400 ms
    assert np.array_equal(got, want), int(np.count_nonzero(got != want))
