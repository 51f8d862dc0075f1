"""Build ``libgdn.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles to an object in parallel, then
one shared library is linked (static CUDA runtime).  Rebuilds only what is
older than its source or the headers.  Usage: ``python -m
gated_delta_rule_49_gb300.build`` or ``build()`` from Python.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
# the debug variant: device-side index and coordinate checks in the prefill
# kernels (-DGDN_BOUNDS_CHECK), same C ABI
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libgdn_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")


def _flags(extra=()):
    return ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-I", INCLUDE, "-I", CSRC,
            "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr", *extra]


def _newest_header() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          bounds_check: bool = False) -> str:
    """Build libgdn.so (or, with bounds_check, libgdn_bounds.so: the same
    library with the device-side index checks of the debug build)."""
    bdir, lib = (BUILD_BOUNDS, LIB_BOUNDS) if bounds_check else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr = _newest_header()
    jobs = []
    objs = []
    for s in srcs:
        obj = os.path.join(bdir, os.path.basename(s)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_info or not os.path.exists(obj) or \
                os.path.getmtime(obj) < max(os.path.getmtime(s), hdr):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            if bounds_check:
                extra.append("-DGDN_BOUNDS_CHECK")
            jobs.append([nvcc(), *_flags(extra), "-c", s, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_info or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if jobs or not os.path.exists(lib) or os.path.getmtime(lib) < max(map(os.path.getmtime, objs)):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-lcuda"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                bounds_check="--bounds-check" in sys.argv))
