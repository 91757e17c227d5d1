"""Builds libmoe.so (the C-ABI library) in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object file
in _build/, then linked into _lib/libmoe.so.  Run as a script or call
``build_library()``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libmoe.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
           "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout)
    if r.stdout.strip():
        sys.stderr.write(r.stdout)


def build_library(extra_flags: list[str] | None = None, verbose: bool = False, lib_path: str = LIB,
                  build_dir: str = BUILD) -> str:
    """Compile csrc/*.cu and link a library (libmoe.so unless lib_path says
    otherwise; a variant with other flags takes its own build_dir); returns
    the library path."""
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    flags = NVFLAGS + (extra_flags or [])
    if verbose:
        flags = flags + ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        _run([nvcc, *ARCH, *flags, "-c", src, "-o", obj])
        return obj

    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"])
    os.replace(tmp, lib_path)
    return lib_path


# A test-only variant: every bounded device wait of the expert kernel gives
# up after 1 ms instead of 2 s, and moe_test_unreachable_wait(1) makes the
# first down unit of the first tile wait for a readiness count that is never
# reached, so that the wait runs out.  Never the library the benchmark or a
# user loads.
WAIT_TEST_LIB = os.path.join(LIBDIR, "libmoe_waittest.so")


def build_wait_test_library() -> str:
    return build_library(["-DMOE_WAIT_TEST"], lib_path=WAIT_TEST_LIB,
                         build_dir=os.path.join(PKG, "_build_waittest"))


if __name__ == "__main__":
    print(build_library(verbose="-v" in sys.argv))
