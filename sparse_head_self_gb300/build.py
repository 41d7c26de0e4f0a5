"""Build libfibatt.so in-tree with nvcc for sm_103a.

Every translation unit under ``csrc/`` is compiled in parallel into
``_build/`` and linked into ``_build/libfibatt.so`` (CUDA runtime linked
statically, no torch dependency).  A unit is rebuilt when it or any header
under ``csrc/`` or ``include/`` is newer than its object.

``build_library(checks=True)`` builds the same sources with
``-DFIBATT_CHECKS`` into ``_build_checks/libfibatt.so``: the debug library
whose kernels check the bounds of their shared-memory stages, windows and
scratch rows and record a failure in the device error word instead of
making the access.  ``FIBATT_CHECKS=1`` in the environment makes the
binding load it.
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
LIB = os.path.join(BUILD, "libfibatt.so")
BUILD_CHECKS = os.path.join(PKG, "_build_checks")
LIB_CHECKS = os.path.join(BUILD_CHECKS, "libfibatt.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libfibatt needs the CUDA toolkit to build")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _compile(args):
    cmd, obj = args
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {obj}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build_library(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
                  checks: bool = False) -> str:
    """Compile and link libfibatt.so (the checks build with checks=True);
    returns its path."""
    build_dir, lib_path = (BUILD_CHECKS, LIB_CHECKS) if checks else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DFIBATT_CHECKS"] if checks else [])
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    hdr_time = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    jobs, objs = [], []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        stale = (force or not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(src)
                 or os.path.getmtime(obj) < hdr_time)
        if stale:
            cmd = [nvcc, *ARCH, *flags, "-I", os.path.join(ROOT, "include"), "-c", src, "-o", obj]
            if ptxas_verbose and src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"]
            jobs.append((cmd, obj))
    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for (cmd, obj), err in zip(jobs, ex.map(_compile, jobs)):
                if verbose and err:
                    print(f"[{os.path.basename(obj)}]\n{err}", file=sys.stderr)
    newest = max(os.path.getmtime(o) for o in objs)
    if force or jobs or not os.path.exists(lib_path) or os.path.getmtime(lib_path) < newest:
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


def build_all(force: bool = False) -> None:
    """The library and its checks build, compiled side by side."""
    with ThreadPoolExecutor(max_workers=2) as ex:
        for f in [ex.submit(build_library, force, False, False, c) for c in (False, True)]:
            f.result()


if __name__ == "__main__":
    checks = "--checks" in sys.argv
    print(build_library(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv, checks=checks))
