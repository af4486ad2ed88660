"""Build libsgemm_gb300.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel to an object file, then linked
into ``dense_fp32_matrix_strict_gb300/_build/libsgemm_gb300.so`` with the
static CUDA runtime. Objects are rebuilt only when a source or header is
newer. ``python -m dense_fp32_matrix_strict_gb300.build`` runs it.

``build(debug=True)`` builds the debug library instead,
``_build_debug/libsgemm_gb300_debug.so``: the same kernels compiled with
``-DSGEMM_DEBUG`` (device-side index and schedule checks that set a status
bit), without the tuning-only families. Set ``SGEMM_LIBRARY`` to its path
to have the binding load it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libsgemm_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_BUILD_DIR, "libsgemm_gb300_debug.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-v",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _deps_mtime() -> float:
    files = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, obj: str, extra=()) -> str:
    log = obj + ".log"
    cmd = [nvcc(), *ARCH_FLAGS, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    with open(log, "w") as f:
        r = subprocess.run(cmd, stdout=f, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        with open(log) as f:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{f.read()}")
    return obj


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every kernel source for sm_103a and link the shared library
    (with debug=True: the debug library, see the module docstring)."""
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    extra = ("-DSGEMM_DEBUG",) if debug else ()
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if debug:
        srcs = [s for s in srcs if not os.path.basename(s).startswith("sgemm_ws_sweep_")]
    dep_t = _deps_mtime()
    jobs = []
    objs = []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(os.path.getmtime(s), dep_t):
            jobs.append((s, o))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for fut in [ex.submit(_compile, s, o, extra) for s, o in jobs]:
                fut.result()
    need_link = force or bool(jobs) or not os.path.exists(lib_path) or any(
        os.path.getmtime(o) > os.path.getmtime(lib_path) for o in objs)
    if need_link:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH_FLAGS, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    if verbose:
        for o in objs:
            log = o + ".log"
            if os.path.exists(log):
                with open(log) as f:
                    sys.stdout.write(f.read())
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
