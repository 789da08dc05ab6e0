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


def build(verbose: bool = False, force: bool = False, extra_flags=None) -> str:
    """Compile and link libdsnq.so; returns its path.  Skips up-to-date work."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    headers = _headers()
    extra = list(extra_flags or [])

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        if force or not _newer(o, [s, *headers, __file__]):
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            if verbose and r.stderr:
                print(r.stderr, file=sys.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    stamp = os.path.join(BUILD_DIR, "libdsnq.stamp")   # which objects the library was linked from
    if force or not _newer(LIB_PATH, objs) or not os.path.exists(stamp) or \
            open(stamp).read() != LIB_PATH + "\n" + platform.machine():
        cmd = [cc, *ARCH, "-shared", "-o", LIB_PATH + ".tmp", *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(LIB_PATH + ".tmp", LIB_PATH)
        with open(stamp, "w") as f:
            f.write(LIB_PATH + "\n" + platform.machine())
    return LIB_PATH


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas-info" in sys.argv else None
    print(build(verbose=v, force="--force" in sys.argv, extra_flags=extra))
