"""The CPU oracle for strict-FP32 SGEMM — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package. The product path (the CUDA library
and its Python binding) never imports, links or calls it, and it shares no
code with that path: the two meet only in the seeded input generator
(``dense_fp32_matrix_strict_gb300.inputs``), which holds none of the
method's arithmetic.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, double accumulation,
OpenMP over rows). It evaluates the plain definition
``C = alpha * A @ B + beta * C0`` ("Optimizing SGEMM in CUDA", section
"What is a SGEMM?"; "The road to a fast GEMM", section "The problem and the
ceiling") and, beside each value, the magnitude sum
``S = |alpha| * sum_k |a_ik b_kj| + |beta c_ij|`` that scales the error bound.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
that do not come from the oracle itself: closed forms (identity, all-ones),
exact integer arithmetic, exact rational brute force, and a hand-worked
example in ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

_lock = threading.Lock()
_lib = None

# Unit roundoff of IEEE-754 binary32 (round to nearest): 2^-24.
U32 = 2.0 ** -24


def build(force: bool = False) -> str:
    """Compile the oracle with gcc + OpenMP into ``oracle/_build``.

    ``-ffp-contract=off`` keeps the compiler from fusing the double
    multiply-adds, so that the oracle's rounding is the same on x86-64 and
    aarch64 hosts.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, f32, vp, ci = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
            lib.oracle_sgemm.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32,
                                         vp, i64, vp, vp, ci]
            lib.oracle_sgemm.restype = ci
            lib.oracle_sgemm_sampled.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64,
                                                 f32, vp, i64, i64, vp, vp, vp, vp, ci]
            lib.oracle_sgemm_sampled.restype = ci
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ci
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads OpenMP gives the oracle when ``nthreads <= 0``."""
    return int(_load().oracle_num_threads())


def _mat(x, rows, cols, name):
    """Return (pointer, leading dimension) of a row-major float32 matrix view."""
    if x is None:
        return None, max(cols, 1)
    x = np.asarray(x)
    if x.dtype != np.float32 or x.ndim != 2 or x.shape != (rows, cols):
        raise ValueError(f"{name}: want float32 array of shape {(rows, cols)}, "
                         f"got {x.dtype} {x.shape}")
    if rows == 0 or cols == 0:
        return x.ctypes.data, max(cols, 1)
    if x.strides[1] != 4 and cols > 1:
        raise ValueError(f"{name}: columns must be contiguous")
    ld = x.strides[0] // 4 if rows > 1 else max(cols, 1)
    return x.ctypes.data, max(ld, cols, 1)


def sgemm_ref(alpha, A, B, beta, C0, nthreads: int = 0):
    """Oracle for every entry: returns ``(ref, S)``, both float64 of shape (M, N).

    ``A`` (M x K), ``B`` (K x N) and ``C0`` (M x N) are float32 arrays whose
    rows may be strided (views into wider buffers); padding is never read.
    ``C0`` may be None when ``beta == 0``.
    """
    A = np.asarray(A)
    B = np.asarray(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    pa, lda = _mat(A, M, K, "A")
    pb, ldb = _mat(B, K, N, "B")
    if C0 is None:
        if beta != 0:
            raise ValueError("C0 is required when beta != 0")
        pc, ldc = None, max(N, 1)
    else:
        pc, ldc = _mat(C0, M, N, "C0")
    ref = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_sgemm(M, N, K, np.float32(alpha), pa, lda, pb, ldb,
                              np.float32(beta), pc, ldc, ref.ctypes.data,
                              S.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm failed ({rc})")
    return ref, S


def sgemm_ref_sampled(alpha, A, B, beta, C0, rows, cols, nthreads: int = 0):
    """Oracle at the entries ``(rows[e], cols[e])``: returns ``(ref, S)`` 1-D."""
    A = np.asarray(A)
    B = np.asarray(B)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    pa, lda = _mat(A, M, K, "A")
    pb, ldb = _mat(B, K, N, "B")
    if C0 is None:
        if beta != 0:
            raise ValueError("C0 is required when beta != 0")
        pc, ldc = None, max(N, 1)
    else:
        pc, ldc = _mat(C0, M, N, "C0")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D of equal length")
    n = rows.shape[0]
    ref = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    rc = _load().oracle_sgemm_sampled(M, N, K, np.float32(alpha), pa, lda, pb, ldb,
                                      np.float32(beta), pc, ldc, n, rows.ctypes.data,
                                      cols.ctypes.data, ref.ctypes.data, S.ctypes.data,
                                      int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm_sampled failed ({rc})")
    return ref, S


def error_bound(K: int, S):
    """Per-element tolerance ``4 * K * 2^-24 * S + 1e-6``.

    This is the forward error bound of a length-K floating-point dot product
    (gamma_K ~ K u with u = 2^-24), widened by a factor 4 to cover the
    epilogue's extra roundings (alpha * acc, beta * c and their sum) and any
    summation order. For K == 0 the result is ``beta * c`` rounded once, so
    K is taken as at least 1.
    """
    return 4.0 * max(int(K), 1) * U32 * np.asarray(S, dtype=np.float64) + 1e-6


def check(C, ref, S, K, exact: bool = False):
    """Compare a float32 result with the oracle.

    ``exact=True`` demands ``C == float32(ref)`` element by element (for
    integer-valued inputs, where every partial sum is exactly representable).
    Otherwise each element must satisfy ``|C - ref| <= error_bound(K, S)``.
    Returns a dict with ``ok``, ``worst`` (max error / bound) and the index
    and values of the worst element.
    """
    C = np.asarray(C, dtype=np.float32)
    ref = np.asarray(ref, dtype=np.float64)
    if C.shape != ref.shape:
        raise ValueError(f"shape mismatch {C.shape} vs {ref.shape}")
    if C.size == 0:
        return {"ok": True, "worst": 0.0, "n": 0}
    if exact:
        want = ref.astype(np.float32)
        bad = ~(C == want)
        nbad = int(np.count_nonzero(bad))
        out = {"ok": nbad == 0, "n": int(C.size), "nbad": nbad, "worst": float(nbad)}
        if nbad:
            idx = np.unravel_index(int(np.argmax(bad)), C.shape)
            out.update(index=tuple(int(i) for i in idx), got=float(C[idx]),
                       want=float(want[idx]))
        return out
    err = np.abs(C.astype(np.float64) - ref)
    tol = error_bound(K, S)
    ratio = np.where(np.isfinite(err), err / tol, np.inf)
    k = int(np.argmax(ratio))
    idx = np.unravel_index(k, C.shape)
    worst = float(ratio[idx])
    return {"ok": bool(worst <= 1.0), "worst": worst, "n": int(C.size),
            "index": tuple(int(i) for i in idx), "got": float(C[idx]),
            "want": float(ref[idx]), "tol": float(tol[idx])}
