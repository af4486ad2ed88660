"""Seeded synthetic inputs for SGEMM tests and benchmarks.

This module holds no SGEMM arithmetic: it only turns (seed, tensor id,
element index) into numbers. It is the one module the CUDA path's tests and
the CPU oracle's tests share.

Generator: splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style. Tensor
``tid`` under ``seed`` has the key ``mix(seed * GAMMA + tid + 1)``; its
element ``e`` (row-major, dense) takes the raw 64-bit draw
``mix(key + (e + 1) * GAMMA)``, i.e. the (e+1)-th output of a splitmix64
stream started at ``key``. Tensor ids: A = 0, B = 1, C0 = 2.

Distributions (the pages show no generator, so these are this library's
own):
  * ``uniform``: ``(z >> 40) * 2^-23 - 1``, a multiple of 2^-23 in
    [-1, 1 - 2^-23]; exact in float32.
  * ``int``:     ``floor(9 * (z >> 11) / 2^53) - 4``, uniform on {-4..4}.
  * ``normal``:  Box-Muller on two draws ``z1 = raw[2e]``, ``z2 = raw[2e+1]``:
    ``sigma * sqrt(-2 ln u1) * cos(2 pi u2)`` with ``u1 = ((z1 >> 11) + 1)
    2^-53`` and ``u2 = (z2 >> 11) 2^-53``, evaluated in float64, then rounded
    to float32.
  * ``zeros``:   all zero.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TID_A, TID_B, TID_C = 0, 1, 2
TID_ROWS, TID_COLS = 10, 11


def _mix(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GAMMA + np.uint64(tid + 1)
    return np.uint64(_mix(np.array([s], dtype=np.uint64))[0])


def raw(seed: int, tid: int, n: int, offset: int = 0, chunk: int = 1 << 24) -> np.ndarray:
    """The ``n`` raw 64-bit draws ``offset .. offset+n-1`` of stream (seed, tid)."""
    key = stream_key(seed, tid)
    out = np.empty(n, dtype=np.uint64)
    for s in range(0, n, chunk):
        e = np.arange(offset + s + 1, offset + min(n, s + chunk) + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            out[s:s + e.shape[0]] = _mix(key + e * GAMMA)
    return out


def _uniform(z):
    return ((z >> np.uint64(40)).astype(np.float64) * 2.0 ** -23 - 1.0).astype(np.float32)


def _int9(z):
    q = ((z >> np.uint64(11)) * np.uint64(9)) >> np.uint64(53)
    return (q.astype(np.int64) - 4).astype(np.float32)


def fill(dist: str, seed: int, tid: int, rows: int, cols: int, sigma: float = 1.0,
         chunk: int = 1 << 22) -> np.ndarray:
    """A dense row-major float32 (rows x cols) matrix from stream (seed, tid).

    Element e depends only on (seed, tid, e), so chunks are generated
    independently, on several host threads for large matrices (numpy releases
    the interpreter lock inside its array operations); the values do not
    depend on the chunking or the thread count.
    """
    if dist not in ("zeros", "uniform", "int", "normal"):
        raise ValueError(f"unknown distribution {dist!r}")
    n = rows * cols
    out = np.empty(n, dtype=np.float32)
    if dist == "zeros":
        out[:] = 0.0
        return out.reshape(rows, cols)

    def one(s):
        m = min(n, s + chunk) - s
        if dist == "uniform":
            out[s:s + m] = _uniform(raw(seed, tid, m, offset=s))
        elif dist == "int":
            out[s:s + m] = _int9(raw(seed, tid, m, offset=s))
        else:
            z = raw(seed, tid, 2 * m, offset=2 * s)
            u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
            u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
            out[s:s + m] = (sigma * np.sqrt(-2.0 * np.log(u1))
                            * np.cos(2.0 * np.pi * u2)).astype(np.float32)

    starts = range(0, n, chunk)
    if n <= chunk:
        for s in starts:
            one(s)
    else:
        workers = max(1, min(16, os.cpu_count() or 1, len(starts)))
        with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, starts))
    return out.reshape(rows, cols)


def sample_entries(M: int, N: int, n: int = 65536, seed: int = 0xC0FFEE):
    """Entries checked on shapes too large for the full oracle.

    ``n`` seeded draws over [0, M) x [0, N) (rows from stream (seed, 10),
    columns from stream (seed, 11), each ``(z >> 32) * size >> 32``), plus
    every entry of the last row and the last column and the four corners.
    Duplicates are removed; the order is row-major.
    """
    if M == 0 or N == 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    zr = raw(seed, TID_ROWS, n) >> np.uint64(32)
    zc = raw(seed, TID_COLS, n) >> np.uint64(32)
    r = ((zr * np.uint64(M)) >> np.uint64(32)).astype(np.int64)
    c = ((zc * np.uint64(N)) >> np.uint64(32)).astype(np.int64)
    last_r = np.full(N, M - 1, np.int64), np.arange(N, dtype=np.int64)
    last_c = np.arange(M, dtype=np.int64), np.full(M, N - 1, np.int64)
    corners = (np.array([0, 0, M - 1, M - 1], np.int64),
               np.array([0, N - 1, 0, N - 1], np.int64))
    rr = np.concatenate([r, last_r[0], last_c[0], corners[0]])
    cc = np.concatenate([c, last_r[1], last_c[1], corners[1]])
    lin = np.unique(rr * N + cc)
    return lin // N, lin % N


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic SGEMM problem: shape, scalars, distributions, seed."""
    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    dist_a: str
    dist_b: str
    dist_c: str
    seed: int
    sigma_a: float = 1.0
    sigma_b: float = 1.0
    sigma_c: float = 1.0
    exact: bool = False          # integer-valued: bit-exact comparison
    full_check: bool = True      # oracle on every entry (else sampled)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def make(self, lda=None, ldb=None, ldc=None):
        """Generate (A, B, C0) as float32 arrays; ld > width gives strided views.

        The logical values never depend on the leading dimensions; padding is
        filled with NaN so that a read of it shows up in the result.
        """
        def padded(vals, rows, cols, ld):
            if ld is None or ld == cols:
                return vals
            buf = np.full((rows, ld), np.nan, dtype=np.float32)
            buf[:, :cols] = vals
            return buf[:, :cols]
        A = fill(self.dist_a, self.seed, TID_A, self.M, self.K, self.sigma_a)
        B = fill(self.dist_b, self.seed, TID_B, self.K, self.N, self.sigma_b)
        C = fill(self.dist_c, self.seed, TID_C, self.M, self.N, self.sigma_c)
        return (padded(A, self.M, self.K, lda), padded(B, self.K, self.N, ldb),
                padded(C, self.M, self.N, ldc))


# The five workloads the library is measured on, in order. Seeds: 0 for the
# first, then 1, 2, 3, 4.
WORKLOADS = {
    "sq256_uniform": Workload("sq256_uniform", 256, 256, 256, 1.0, 0.0,
                              "uniform", "uniform", "uniform", seed=0),
    "sq1024_int": Workload("sq1024_int", 1024, 1024, 1024, 2.0, -1.0,
                           "int", "int", "int", seed=1, exact=True),
    "sq4096_uniform": Workload("sq4096_uniform", 4096, 4096, 4096, 1.0, 0.0,
                               "uniform", "uniform", "uniform", seed=2),
    "ragged_4093x5120x1531_normal": Workload(
        "ragged_4093x5120x1531_normal", 4093, 5120, 1531, 0.7, -1.3,
        "normal", "normal", "normal", seed=3),
    "llm_8192x14336x4096": Workload(
        "llm_8192x14336x4096", 8192, 14336, 4096, 1.0, 0.0,
        "normal", "normal", "zeros", seed=4, sigma_b=0.02, full_check=False),
}
