"""Builds the in-tree shared libraries for sm_103a with nvcc.

libzero3.so        -- the C ABI (include/zero3.h): planner, kernels, launches
libzero3_synth.so  -- the device side of the seeded input generator

Translation units compile in parallel; a library is rebuilt only when a
source or header is newer than it.  Host code is compiled with
-ffp-contract=off and device code with -fmad=false so that no multiply-add is
contracted anywhere.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
          "-Xcompiler", "-ffp-contract=off", "-Xcompiler", "-fno-fast-math",
          f"-I{INCLUDE}"]

LIBS = {
    "libzero3.so": ["plan.cpp", "api.cpp", "checkpoint.cpp", "coordinator.cpp", "kernels.cu",
                    "pieces.cu"],
    "libzero3_synth.so": ["synth.cu"],
}
HEADERS = [os.path.join(CSRC, "internal.h"), os.path.join(CSRC, "device_common.cuh"),
           os.path.join(INCLUDE, "zero3.h")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero3")


def lib_path(name: str) -> str:
    return os.path.join(PKG, name)


def _stale(target: str, sources) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _run(cmd, log):
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout)
    if r.returncode != 0:
        raise RuntimeError(f"build failed: {' '.join(cmd)}\n{r.stdout}")
    return r.stdout


def build_all(quiet: bool = False, force: bool = False) -> dict:
    """Compile every library that is missing or out of date; returns paths."""
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    jobs = []
    for lib, srcs in LIBS.items():
        paths = [os.path.join(CSRC, s) for s in srcs]
        if force or _stale(lib_path(lib), paths + HEADERS):
            jobs.append((lib, paths))
    if jobs:
        compiles = []
        for lib, paths in jobs:
            for src in paths:
                obj = os.path.join(BUILD, os.path.basename(src) + ".o")
                cmd = [exe] + ARCH + COMMON + ["-Xptxas", "-v", "-c", src, "-o", obj]
                compiles.append((cmd, obj + ".log"))
        with ThreadPoolExecutor(max_workers=min(8, len(compiles))) as ex:
            list(ex.map(lambda c: _run(*c), compiles))
        for lib, paths in jobs:
            objs = [os.path.join(BUILD, os.path.basename(s) + ".o") for s in paths]
            tmp = lib_path(lib) + ".tmp"
            _run([exe] + ARCH + ["-shared", "-o", tmp] + objs, os.path.join(BUILD, lib + ".log"))
            os.replace(tmp, lib_path(lib))
            if not quiet:
                print(f"built {lib_path(lib)}", file=sys.stderr)
    return {lib: lib_path(lib) for lib in LIBS}


if __name__ == "__main__":
    build_all(force="--force" in sys.argv)
