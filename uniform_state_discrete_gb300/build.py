"""Build the sm_103a shared library ``_build/libdgsampler.so`` in-tree with nvcc.

Each translation unit is compiled in parallel, then linked with the static CUDA
runtime.  ``python uniform_state_discrete_gb300/build.py [-v]`` builds from the
command line (``-v`` prints ptxas register and spill reports); importing the
package itself requires the built library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(BUILD, "libdgsampler.so")
# the same library with index checks and workspace guards (DG_DEBUG_CHECKS), for the debug tests
SO_DEBUG = os.path.join(BUILD, "libdgsampler_debug.so")
SOURCES = ["dg_sampler.cu", "dg_kernels.cu", "dg_lmhead.cu", "dg_static.cu", "dg_selfcond.cu"]
HEADERS = ["dg_internal.cuh", "dg_tail.cuh", "dg_gumbel.cuh", "dg_norm.cuh", "dg_tc.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libdgsampler.so")


def flags(verbose: bool = False, debug: bool = False) -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if debug:
        f += ["-DDG_DEBUG_CHECKS"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(so: str) -> bool:
    if not os.path.exists(so):
        return True
    t = os.path.getmtime(so)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "dg_sampler.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Build the library (``debug``: the index-checking build, ``_build/libdgsampler_debug.so``)."""
    so = SO_DEBUG if debug else SO
    if not (force or _stale(so)):
        return so
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    procs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", "_debug.o" if debug else ".o"))
        cmd = [exe] + flags(verbose, debug) + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    objs, failed = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(f"--- {src}\n{out}")
        if p.returncode:
            failed.append(src)
        objs.append(obj)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = so + f".tmp{os.getpid()}"
    subprocess.run([exe] + ARCH + ["-shared", "-o", tmp] + objs, check=True)
    os.replace(tmp, so)
    return so


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
