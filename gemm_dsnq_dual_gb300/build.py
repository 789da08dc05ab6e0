"""Builds libdsnq.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in its own nvcc process, in parallel, then
linked into a shared library next to this file.  nvcc cross-compiles, so this
runs on hosts without a GPU.  Run as `python -m gemm_dsnq_dual_gb300.build`.
"""

from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
# Objects are kept per host architecture, so a tree copied between an x86
# build host and an Arm GPU host never links foreign objects.
BUILD_DIR = os.path.join(ROOT, "_build", platform.machine() or "unknown")
LIB_NAME = "libdsnq.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libdsnq_debug.so")   # device index checks (DSNQ_DEBUG)

SOURCES = ["norm_quant.cu", "gemm_fp8.cu", "dsnq_api.cu", "static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def _headers():
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _build_one(debug: bool, verbose: bool, force: bool, extra_flags, pool) -> str:
    variant = "debug" if debug else "release"
    bdir = os.path.join(BUILD_DIR, variant)
    os.makedirs(bdir, exist_ok=True)
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    cc = nvcc()
    headers = _headers()
    extra = list(extra_flags or []) + (["-DDSNQ_DEBUG"] if debug else [])

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        if force or not _newer(o, [s, *headers, __file__]):
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr, file=sys.stderr)
        return o

    objs = list(pool.map(compile_one, SOURCES))
    stamp = os.path.join(bdir, "libdsnq.stamp")   # which objects the library was linked from
    if force or not _newer(lib_path, objs) or not os.path.exists(stamp) or \
            open(stamp).read() != lib_path + "\n" + platform.machine():
        cmd = [cc, *ARCH, "-shared", "-o", lib_path + ".tmp", *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(lib_path + ".tmp", lib_path)
        with open(stamp, "w") as f:
            f.write(lib_path + "\n" + platform.machine())
    return lib_path


def build(verbose: bool = False, force: bool = False, extra_flags=None, debug: bool = True) -> str:
    """Compile and link libdsnq.so (and, with debug=True, libdsnq_debug.so:
    the same sources with the device index checks of DSNQ_DEBUG); returns the
    release library's path.  Skips up-to-date work."""
    # Two builders, each compiling its sources on a shared pool of nvcc jobs
    # (the builders only wait; the compiles run on the other pool).
    with ThreadPoolExecutor(max_workers=2 * len(SOURCES)) as cc_pool, ThreadPoolExecutor(max_workers=2) as libs:
        jobs = [libs.submit(_build_one, False, verbose, force, extra_flags, cc_pool)]
        if debug:
            jobs.append(libs.submit(_build_one, True, verbose, force, extra_flags, cc_pool))
        paths = [j.result() for j in jobs]
    return paths[0]


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-info" in sys.argv else None
    print(build(verbose=v, force="--force" in sys.argv, extra_flags=extra))
