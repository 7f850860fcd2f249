"""Build ``librlscan.so`` (the CUDA library behind the C ABI) in-tree.

Each translation unit in ``csrc/`` is compiled in parallel with nvcc for
sm_103a only, then linked into ``linear_recurrence_scan_gb300/_build/
librlscan.so``.  Run ``python -m linear_recurrence_scan_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "librlscan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", CSRC, "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librlscan")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return (sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) +
            [os.path.join(INCLUDE, "rlscan.h")])


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


CHECKED_DIR = os.path.join(OUT_DIR, "checked")


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str = OUT_DIR) -> str:
    """Compile and link the library into ``out_dir``; returns its path.
    Rebuilds only when a source or header is newer than the library (or
    ``force``)."""
    lib_path = os.path.join(out_dir, "librlscan.so")
    srcs = _sources()
    deps = srcs + _headers() + [os.path.abspath(__file__)]
    if not force and not _stale(lib_path, deps):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_checked(force: bool = False) -> str:
    """The bounds-checked build (RLSCAN_CHECK_BOUNDS=1: every global access
    and bulk copy of the scan kernels is tested against its argument's
    extent, violations are counted and skipped), in its own directory."""
    return build(force, extra_flags=("-DRLSCAN_CHECK_BOUNDS=1",), out_dir=CHECKED_DIR)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else ()))
