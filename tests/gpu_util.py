"""Helpers for the GPU parity tests: place seeded host matrices on the device
with chosen leading dimensions, base offsets and NaN guard bands, call the
library through its C ABI, and read back C plus the guard bands."""
from __future__ import annotations

import numpy as np

import dense_fp32_matrix_strict_gb300 as sg

GUARD = 64          # floats of NaN before and after every matrix


def _torch():
    import torch
    return torch


def place(x, ld=None, offset=0, pad_value=np.nan):
    """Copy host matrix x (rows x cols) into a fresh device buffer.

    Layout: GUARD + offset floats of pad, then rows of length ld (the
    padding columns hold pad_value), then GUARD floats of pad. Returns
    (view, buffer, start) where view is the (rows x cols) strided tensor.
    """
    torch = _torch()
    rows, cols = x.shape
    ld = max(ld or cols, cols, 1)
    start = GUARD + offset
    n = start + rows * ld + GUARD
    buf = torch.full((n,), float(pad_value), dtype=torch.float32, device="cuda")
    mat = buf[start:start + rows * ld].view(rows, ld)
    view = mat[:, :cols]
    if rows and cols:
        view.copy_(torch.from_numpy(np.ascontiguousarray(x)).to("cuda"))
    return view, buf, start


def untouched_outside(buf, start, rows, cols, ld, pad_value=np.nan):
    """True if every float of buf outside the rows x cols window is still pad."""
    host = buf.cpu().numpy()
    mask = np.ones(host.shape, dtype=bool)
    ld = max(ld, cols, 1)
    for r in range(rows):
        mask[start + r * ld:start + r * ld + cols] = False
    rest = host[mask]
    if np.isnan(pad_value):
        return bool(np.all(np.isnan(rest)))
    return bool(np.all(rest == pad_value))


def run(alpha, A, B, beta, C0, lda=None, ldb=None, ldc=None, offsets=(0, 0, 0),
        stream=None, c_fill=None, transa=False, transb=False):
    """Run sgemm on device copies of A, B, C0; return (C, guards_ok, plan).

    With transa / transb, A / B are the stored matrices (K x M / N x K) and
    the call computes alpha * op(A) op(B) + beta * C through sgemm_ex.

    C0 None means C starts as NaN (only valid when beta == 0, which must not
    read C); c_fill overrides C's starting contents likewise.
    """
    torch = _torch()
    M = A.shape[1] if transa else A.shape[0]
    N = B.shape[0] if transb else B.shape[1]
    dA, _, _ = place(A, lda, offsets[0])
    dB, _, _ = place(B, ldb, offsets[1])
    start_c = C0 if C0 is not None else np.full((M, N), np.nan if c_fill is None else c_fill,
                                                np.float32)
    dC, bufC, startC = place(start_c, ldc, offsets[2])
    plan = sg.plan_tensors(alpha, dA, dB, beta, dC, transa=transa, transb=transb)
    sg.sgemm_tensors(alpha, dA, dB, beta, dC, stream=stream, transa=transa, transb=transb)
    sg.check_status(stream=stream)
    torch.cuda.synchronize()
    C = dC.cpu().numpy()
    ok = untouched_outside(bufC, startC, M, N, max(ldc or N, N, 1))
    return C, ok, plan
