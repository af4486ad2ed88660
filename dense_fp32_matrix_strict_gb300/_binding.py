"""ctypes binding of ``libsgemm_gb300.so`` — argument marshalling only.

Each function here has the name and argument order of the C entry point in
``include/sgemm.h``. All arithmetic happens in the CUDA kernels; there is no
CPU path. If the shared library has not been built, every call raises
``RuntimeError`` (build it with ``dense_fp32_matrix_strict_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SGEMM_OK = 0
SGEMM_ERR_INVALID_VALUE = 1
SGEMM_ERR_UNSUPPORTED_DEVICE = 2
SGEMM_ERR_LAUNCH = 3
SGEMM_ERR_DEVICE_TIMEOUT = 4
SGEMM_ERR_CUDA = 5
SGEMM_ERR_DEVICE_CHECK = 6

# Every function include/sgemm.h declares.
EXPORTED_SYMBOLS = (
    "sgemm", "sgemm_check_status", "sgemm_error_string", "sgemm_last_cuda_error",
    "sgemm_plan", "sgemm_set_config", "sgemm_set_wait_timeout_ns", "sgemm_fp32_peak",
    "sgemm_selftest_wait_timeout", "sgemm_config_names", "sgemm_noalloc", "sgemm_3xtf32",
    "sgemm_set_shape_config", "sgemm_clear_shape_configs", "sgemm_ex", "sgemm_plan_ex",
    "sgemm_3xtf32_ex", "sgemm_host", "sgemm_noalloc_check_status", "sgemm_fp32_peak_ex",
    "sgemm_null_launch", "sgemm_tf32_mma_peak", "sgemm_selftest_occupy",
)

SGEMM_PEAK_FFMA, SGEMM_PEAK_FFMA2, SGEMM_PEAK_OUTER = 0, 1, 2

SGEMM_OP_N, SGEMM_OP_T = 0, 1

_lock = threading.Lock()
_lib = None


class SgemmError(RuntimeError):
    """A non-zero return code from the library."""

    def __init__(self, func: str, code: int):
        self.code = int(code)
        msg = _lib.sgemm_error_string(code).decode() if _lib is not None else str(code)
        cuda = _lib.sgemm_last_cuda_error() if _lib is not None else 0
        extra = f" (CUDA error {cuda})" if cuda and code in (SGEMM_ERR_LAUNCH, SGEMM_ERR_CUDA) else ""
        super().__init__(f"{func} failed: {msg} [code {code}]{extra}")


def library_path() -> str:
    return os.environ.get("SGEMM_LIBRARY") or _build.LIB_PATH


def load():
    """Load the shared library (once). Raises RuntimeError if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # SGEMM_LIBRARY selects another build of the same library (the
        # debug build, for instance); by default the in-tree release build.
        path = os.environ.get("SGEMM_LIBRARY") or _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: the CUDA library has not been built "
                "(run `python -m dense_fp32_matrix_strict_gb300.build`); there is no CPU path")
        lib = ctypes.CDLL(path)
        i64, f32, vp, ci, f64p = (ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.POINTER(ctypes.c_double))
        lib.sgemm.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm.restype = ci
        lib.sgemm_check_status.argtypes = [vp, ctypes.POINTER(ci)]
        lib.sgemm_check_status.restype = ci
        lib.sgemm_error_string.argtypes = [ci]
        lib.sgemm_error_string.restype = ctypes.c_char_p
        lib.sgemm_last_cuda_error.argtypes = []
        lib.sgemm_last_cuda_error.restype = ci
        lib.sgemm_plan.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                   ctypes.c_char_p, ci, ctypes.POINTER(ci)]
        lib.sgemm_plan.restype = ci
        lib.sgemm_set_config.argtypes = [ctypes.c_char_p]
        lib.sgemm_set_config.restype = ci
        lib.sgemm_config_names.argtypes = [ctypes.c_char_p, ci]
        lib.sgemm_config_names.restype = ci
        lib.sgemm_set_shape_config.argtypes = [i64, i64, i64, ctypes.c_char_p]
        lib.sgemm_set_shape_config.restype = ci
        lib.sgemm_clear_shape_configs.argtypes = []
        lib.sgemm_clear_shape_configs.restype = ci
        lib.sgemm_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.sgemm_set_wait_timeout_ns.restype = ci
        lib.sgemm_fp32_peak.argtypes = [ctypes.c_double, f64p, f64p, f64p, vp]
        lib.sgemm_fp32_peak.restype = ci
        lib.sgemm_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.sgemm_selftest_wait_timeout.restype = ci
        lib.sgemm_selftest_occupy.argtypes = [ci, ctypes.c_uint64, vp]
        lib.sgemm_selftest_occupy.restype = ci
        lib.sgemm_noalloc.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_noalloc.restype = ci
        lib.sgemm_noalloc_check_status.argtypes = [vp, ctypes.POINTER(ci)]
        lib.sgemm_noalloc_check_status.restype = ci
        lib.sgemm_fp32_peak_ex.argtypes = [ci, ctypes.c_double, f64p, f64p, f64p, vp]
        lib.sgemm_fp32_peak_ex.restype = ci
        lib.sgemm_null_launch.argtypes = [vp]
        lib.sgemm_tf32_mma_peak.argtypes = [ci, ctypes.c_double, f64p, f64p, f64p, vp]
        lib.sgemm_tf32_mma_peak.restype = ci
        lib.sgemm_null_launch.restype = ci
        lib.sgemm_3xtf32.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_3xtf32.restype = ci
        lib.sgemm_ex.argtypes = [ci, ci, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_ex.restype = ci
        lib.sgemm_3xtf32_ex.argtypes = [ci, ci, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp,
                                        i64, vp]
        lib.sgemm_3xtf32_ex.restype = ci
        lib.sgemm_plan_ex.argtypes = [ci, ci, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                      ctypes.c_char_p, ci, ctypes.POINTER(ci)]
        lib.sgemm_plan_ex.restype = ci
        lib.sgemm_host.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.sgemm_host.restype = ci
        _lib = lib
        return lib


def _check(func: str, rc: int) -> int:
    if rc != SGEMM_OK:
        raise SgemmError(func, rc)
    return rc


# ---- raw entry points (same names and argument order as the C ABI) --------

def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """C = alpha*A*B + beta*C on device pointers (ints); returns the raw code."""
    return load().sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """sgemm without any device allocation (fixed scratch inside the library);
    device pointers as ints; returns the raw code."""
    return load().sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_noalloc_check_status(stream=0):
    """Returns (code, bits) of the scratch status word sgemm_noalloc writes."""
    bits = ctypes.c_int(0)
    rc = load().sgemm_noalloc_check_status(stream, ctypes.byref(bits))
    return rc, bits.value


def sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """The tcgen05 3xTF32 path (device pointers as ints); returns the raw code."""
    return load().sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """C = alpha*op(A)*op(B) + beta*C (op: SGEMM_OP_N / SGEMM_OP_T); raw code."""
    return load().sgemm_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_3xtf32_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().sgemm_3xtf32_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_plan_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc):
    """Returns (code, kernel name, grid)."""
    buf = ctypes.create_string_buffer(128)
    grid = ctypes.c_int(0)
    rc = load().sgemm_plan_ex(opa, opb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, buf, 128,
                              ctypes.byref(grid))
    return rc, buf.value.decode(), grid.value


def sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """C = alpha*A*B + beta*C with HOST pointers (ints); returns the raw code."""
    return load().sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def sgemm_check_status(stream=0):
    """Returns (code, bits)."""
    bits = ctypes.c_int(0)
    rc = load().sgemm_check_status(stream, ctypes.byref(bits))
    return rc, bits.value


def sgemm_error_string(code: int) -> str:
    return load().sgemm_error_string(code).decode()


def sgemm_last_cuda_error() -> int:
    return load().sgemm_last_cuda_error()


def sgemm_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc):
    """Returns (code, kernel name, grid)."""
    buf = ctypes.create_string_buffer(128)
    grid = ctypes.c_int(0)
    rc = load().sgemm_plan(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, buf, 128,
                           ctypes.byref(grid))
    return rc, buf.value.decode(), grid.value


def sgemm_set_config(name: str) -> int:
    return load().sgemm_set_config(name.encode())


def sgemm_set_shape_config(M: int, N: int, K: int, name) -> int:
    """Per-shape configuration rule; name None or "auto" removes it."""
    return load().sgemm_set_shape_config(M, N, K, None if name is None else name.encode())


def sgemm_clear_shape_configs() -> int:
    return load().sgemm_clear_shape_configs()


def sgemm_config_names():
    """Returns (code, [family names])."""
    buf = ctypes.create_string_buffer(4096)
    rc = load().sgemm_config_names(buf, 4096)
    names = buf.value.decode().split(",") if rc == SGEMM_OK and buf.value else []
    return rc, names


def sgemm_set_wait_timeout_ns(ns: int) -> int:
    return load().sgemm_set_wait_timeout_ns(int(ns))


def sgemm_fp32_peak(target_ms: float = 200.0, stream=0):
    """Returns (code, gflops, ms, flops)."""
    g, m, f = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    rc = load().sgemm_fp32_peak(float(target_ms), ctypes.byref(g), ctypes.byref(m),
                                ctypes.byref(f), stream)
    return rc, g.value, m.value, f.value


def sgemm_fp32_peak_ex(form: int, target_ms: float = 200.0, stream=0):
    """Returns (code, gflops, ms, flops) of the chosen instruction form."""
    g, m, f = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    rc = load().sgemm_fp32_peak_ex(int(form), float(target_ms), ctypes.byref(g),
                                   ctypes.byref(m), ctypes.byref(f), stream)
    return rc, g.value, m.value, f.value


def sgemm_tf32_mma_peak(n: int = 128, target_ms: float = 100.0, stream=0):
    """Returns (code, tflops, ms, flops) of the TF32 tcgen05 MMA ceiling."""
    t, m, f = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
    rc = load().sgemm_tf32_mma_peak(int(n), float(target_ms), ctypes.byref(t), ctypes.byref(m),
                                    ctypes.byref(f), stream)
    return rc, t.value, m.value, f.value


def sgemm_null_launch(stream=0) -> int:
    """One empty kernel on `stream` (the launch-latency floor); raw code."""
    return load().sgemm_null_launch(stream)


def sgemm_selftest_wait_timeout(timeout_ns: int, stream=0) -> int:
    return load().sgemm_selftest_wait_timeout(int(timeout_ns), stream)


def sgemm_selftest_occupy(ctas: int, ns: int, stream=0) -> int:
    """`ctas` CTAs holding one SM each for `ns` ns on `stream`; raw code."""
    return load().sgemm_selftest_occupy(int(ctas), int(ns), stream)


# ---- torch tensor convenience (marshalling only) --------------------------

def _ld(t, rows, cols, name):
    import torch
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dim() != 2 or tuple(t.shape) != (rows, cols):
        raise ValueError(f"{name} must have shape {(rows, cols)}, got {tuple(t.shape)}")
    if rows == 0 or cols == 0:
        return max(cols, 1)
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with contiguous columns")
    return max(t.stride(0) if rows > 1 else cols, cols, 1)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        idx = device.index if hasattr(device, "index") else device
        if idx is None:
            idx = torch.cuda.current_device()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return int(raw(idx))
        stream = torch.cuda.current_stream(idx)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


class _on_device:
    """Make `device` current for the duration of a call (no-op if it is)."""

    def __init__(self, device):
        import torch
        self.idx = device.index if device.index is not None else torch.cuda.current_device()
        self.prev = None

    def __enter__(self):
        import torch
        cur = torch.cuda.current_device()
        if cur != self.idx:
            self.prev = cur
            torch.cuda.set_device(self.idx)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            import torch
            torch.cuda.set_device(self.prev)
        return False


def _shapes(A, B, transa, transb):
    """(M, N, K, lda, ldb) of op(A) op(B) from the stored tensors."""
    M, K = (A.shape[1], A.shape[0]) if transa else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if transb else (B.shape[0], B.shape[1])
    if K2 != K:
        raise ValueError(f"inner dimensions differ: op(A) is {(M, K)}, op(B) is {(K2, N)}")
    lda = _ld(A, A.shape[0], A.shape[1], "A")
    ldb = _ld(B, B.shape[0], B.shape[1], "B")
    return M, N, K, lda, ldb


def _op(flag: bool) -> int:
    return SGEMM_OP_T if flag else SGEMM_OP_N


def sgemm_tensors(alpha, A, B, beta, C, stream=None, transa=False, transb=False) -> None:
    """C = alpha * op(A) @ op(B) + beta * C in place on row-major float32 CUDA tensors.

    op(X) is X, or X.T when trans* is set (the tensor is then the stored,
    untransposed matrix: A of shape (K, M), B of shape (N, K)). Rows may be
    strided (leading dimension = stride(0)). Launches on ``stream``
    (default: torch's current stream on C's device). Raises SgemmError on a
    non-zero return code.
    """
    M, N, K, lda, ldb = _shapes(A, B, transa, transb)
    ldc = _ld(C, M, N, "C")
    if not (A.device == B.device == C.device):
        raise ValueError("A, B and C must be on the same device")
    with _on_device(C.device):
        h = _stream_handle(stream, C.device)
        if transa or transb:
            rc = load().sgemm_ex(_op(transa), _op(transb), M, N, K, float(alpha), A.data_ptr(),
                                 lda, B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc, h)
        else:
            rc = load().sgemm(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                              float(beta), C.data_ptr(), ldc, h)
    if rc != SGEMM_OK:
        raise SgemmError("sgemm_ex" if (transa or transb) else "sgemm", rc)


def sgemm_3xtf32_tensors(alpha, A, B, beta, C, stream=None, transa=False, transb=False) -> None:
    """sgemm_tensors through the tcgen05 3xTF32 entry points."""
    M, N, K, lda, ldb = _shapes(A, B, transa, transb)
    ldc = _ld(C, M, N, "C")
    with _on_device(C.device):
        h = _stream_handle(stream, C.device)
        if transa or transb:
            rc = load().sgemm_3xtf32_ex(_op(transa), _op(transb), M, N, K, float(alpha),
                                        A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
                                        C.data_ptr(), ldc, h)
        else:
            rc = load().sgemm_3xtf32(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                                     float(beta), C.data_ptr(), ldc, h)
    if rc != SGEMM_OK:
        raise SgemmError("sgemm_3xtf32", rc)


def _host_ld(t, rows, cols, name):
    import torch
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.is_cuda:
        raise TypeError(f"{name} must be a host (CPU) tensor")
    if t.dim() != 2 or tuple(t.shape) != (rows, cols):
        raise ValueError(f"{name} must have shape {(rows, cols)}, got {tuple(t.shape)}")
    if rows == 0 or cols == 0:
        return max(cols, 1)
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with contiguous columns")
    return max(t.stride(0) if rows > 1 else cols, cols, 1)


def sgemm_host_tensors(alpha, A, B, beta, C, stream=None, device=None) -> None:
    """sgemm_host on row-major float32 CPU tensors (pin them for overlap).

    Enqueued on ``stream`` (default: torch's current stream on ``device``);
    C is complete once that stream is synchronised.
    """
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    lda = _host_ld(A, M, K, "A")
    ldb = _host_ld(B, K, N, "B")
    ldc = _host_ld(C, M, N, "C")
    dev = (torch.device("cuda", torch.cuda.current_device()) if device is None
           else torch.device(device))
    with _on_device(dev):
        rc = load().sgemm_host(M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb,
                               float(beta), C.data_ptr(), ldc, _stream_handle(stream, dev))
    if rc != SGEMM_OK:
        raise SgemmError("sgemm_host", rc)


def plan_tensors(alpha, A, B, beta, C, transa=False, transb=False):
    """Kernel name and grid sgemm_tensors would use for these tensors."""
    M, N, K, lda, ldb = _shapes(A, B, transa, transb)
    with _on_device(C.device):
        rc, name, grid = sgemm_plan_ex(_op(transa), _op(transb), M, N, K, float(alpha),
                                       A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
                                       C.data_ptr(), _ld(C, M, N, "C"))
    _check("sgemm_plan_ex", rc)
    return name, grid


def check_status(stream=None, device=None) -> int:
    """Synchronise and read/clear the device status word; raise on a time-out."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        rc, bits = sgemm_check_status(_stream_handle(stream, dev))
    _check("sgemm_check_status", rc)
    return bits


def fp32_peak(target_ms: float = 200.0, stream=None, device=None, form: int = SGEMM_PEAK_FFMA):
    """Measured FP32 ceiling in one instruction form (SGEMM_PEAK_FFMA,
    SGEMM_PEAK_FFMA2, or SGEMM_PEAK_OUTER: the GEMM's register outer product
    without its loads): dict(gflops, ms, flops)."""
    import torch
    dev = device if device is not None else torch.cuda.current_device()
    with torch.cuda.device(dev):
        rc, g, m, f = sgemm_fp32_peak_ex(form, target_ms, _stream_handle(stream, dev))
    _check("sgemm_fp32_peak_ex", rc)
    return {"gflops": g, "ms": m, "flops": f}
