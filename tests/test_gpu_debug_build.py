"""The debug build (-DSGEMM_DEBUG): the same kernels with device-side checks
of every shared-memory, workspace and C index and of each work item against
the schedule. A failed check sets a status bit (16) and the kernel carries on,
so the host reads it through sgemm_check_status.

The debug library is built from the same sources (build(debug=True)) and run
in a child process that loads it through SGEMM_LIBRARY, over plans that
reach every kernel family "auto" chooses between, the stream-K tail (finished
in the kernel and by the fixup kernel), cp.async loads, the packing and
transposing copies, transposed operands, clusters, k-groups, the
allocation-free entry point and the 3xTF32 kernels. Every case must come
back with a clear status word and within the oracle's bound.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, sys
import numpy as np
import torch
import dense_fp32_matrix_strict_gb300 as sg
import oracle
from dense_fp32_matrix_strict_gb300 import inputs
from tests import gpu_util

assert sg.library_path().endswith("libsgemm_gb300_debug.so"), sg.library_path()
CASES = [
    # (config, M, N, K, lda, ldb, ldc, offsets, transa, transb, entry)
    ("auto", 300, 260, 200, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 1024, 1024, 1024, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 1000, 1100, 2000, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 1024, 1024, 4096, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 2048, 2048, 4096, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 256, 256, 256, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 512, 512, 512, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 256, 256, 8192, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 130, 70, 4100, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 333, 517, 401, 403, 519, 520, (1, 2, 3), False, False, "sgemm"),
    ("auto", 700, 900, 301, None, None, None, (0, 0, 0), True, True, "sgemm"),
    ("128x128", 1000, 1100, 2000, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("128x128:fixup", 1000, 1100, 2000, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("128x128:cpasync", 333, 4500, 777, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("64x64:cpasync", 129, 127, 31, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("128x64", 513, 640, 96, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("ws_128x64x32_s4_k2", 1024, 1024, 1024, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("ws_64x64x32_s4_k4_c4", 256, 256, 256, None, None, None, (0, 0, 0), False, False, "sgemm"),
    # fewer k-tiles than CTAs in the cluster: some ranks have nothing to add
    ("ws_64x64x32_s4_k4_c4", 70, 90, 20, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("ws_64x64x32_s4_k4_c4:at", 70, 90, 40, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto:xp", 2048, 2048, 2048, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto:atcopy", 1000, 3000, 4000, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 1021, 2600, 3001, None, None, None, (0, 0, 0), False, False, "sgemm"),
    ("auto", 2000, 2100, 1900, None, None, None, (0, 0, 0), True, True, "sgemm"),
    ("128x128", 1000, 1100, 2000, None, None, None, (0, 0, 0), False, False, "noalloc"),
    ("auto", 4096, 4096, 256, None, None, None, (0, 0, 0), False, False, "3xtf32"),
    ("auto", 300, 640, 500, None, None, None, (0, 0, 0), False, False, "3xtf32"),
]
out = []
for i, (cfg, M, N, K, lda, ldb, ldc, offs, ta, tb, entry) in enumerate(CASES):
    assert sg.sgemm_set_config(cfg) == 0, cfg
    sa = (K, M) if ta else (M, K)
    sb = (N, K) if tb else (K, N)
    A = inputs.fill("normal", 700 + i, inputs.TID_A, *sa)
    B = inputs.fill("normal", 700 + i, inputs.TID_B, *sb)
    C0 = inputs.fill("normal", 700 + i, inputs.TID_C, M, N)
    if entry == "sgemm":
        C, guards, plan = gpu_util.run(0.7, A, B, -1.3, C0, lda=lda, ldb=ldb, ldc=ldc,
                                       offsets=offs, transa=ta, transb=tb)
        name = plan[0]
    else:
        dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C0))
        if entry == "noalloc":
            rc = sg.sgemm_noalloc(M, N, K, 0.7, dA.data_ptr(), K, dB.data_ptr(), N, -1.3,
                                  dC.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
            assert rc == 0, rc
            rc, bits = sg.sgemm_noalloc_check_status(torch.cuda.current_stream().cuda_stream)
            assert (rc, bits) == (0, 0), (entry, rc, bits)
        else:
            sg.sgemm_3xtf32_tensors(0.7, dA, dB, -1.3, dC)
        C, guards, name = dC.cpu().numpy(), True, entry
    rc, bits = sg.sgemm_check_status()
    opA = A.T if ta else A
    opB = B.T if tb else B
    ref, S = oracle.sgemm_ref(0.7, np.ascontiguousarray(opA), np.ascontiguousarray(opB), -1.3, C0)
    rep = oracle.check(C, ref, S, K)
    out.append({"case": i, "config": cfg, "plan": name, "rc": rc, "bits": bits,
                "guards": bool(guards), "ok": bool(rep["ok"]), "worst": rep["worst"]})
sg.sgemm_set_config("auto")
print(json.dumps(out))
"""


def test_debug_build_runs_every_plan_with_clear_status():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dense_fp32_matrix_strict_gb300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, SGEMM_LIBRARY=lib, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", _CHILD], env=env, cwd=ROOT, timeout=900,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    results = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(results) == 27
    for res in results:
        assert res["rc"] == 0 and res["bits"] == 0, res
        assert res["guards"] and res["ok"], res
    plans = {res["plan"] for res in results}
    # The debug kernels covered the families and paths listed above.
    for tag in ("+sk", "+skfix", "+packAT", "+packATfused", "+packBT", "+packBTfused", "_c4_",
                "_k2_", "_k4_",
                "_Axp_", "_Acp_",
                "noalloc", "3xtf32"):
        assert any(tag in p for p in plans), (tag, sorted(plans))
