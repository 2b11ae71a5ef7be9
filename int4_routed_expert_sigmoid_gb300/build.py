"""Build libmoe.so (the CUDA library behind include/moe.h) in-tree with nvcc.

Each translation unit under csrc/ is compiled for sm_103a in parallel, then
linked into ``_build/libmoe.so`` with the static CUDA runtime (the library
needs no libcuda at link time; it looks up the one driver call it uses, the
TMA descriptor encoder, at run time).

    python -m int4_routed_expert_sigmoid_gb300.build [--force] [--verbose] [--debug-bounds]

With ``debug_bounds`` the same sources are built with ``MOE_DEBUG_BOUNDS`` into
``_build_debug/libmoe.so``: every index the kernels read another buffer by
(expert id, pair position, token row) is checked, and one out of range sets
MOE_DEVERR_BOUNDS in the call's error word and skips the access.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB = os.path.join(BUILD, "libmoe.so")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libmoe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "moe.h"), os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          debug_bounds: bool = False) -> str:
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if debug_bounds:
        extra.append("-DMOE_DEBUG_BOUNDS")

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log:
                sys.stderr.write(log)
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libmoe.so failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--debug-bounds", action="store_true", help="build the bounds-checked library")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas, debug_bounds=a.debug_bounds))


if __name__ == "__main__":
    main()
