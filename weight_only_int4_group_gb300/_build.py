"""Build libq4.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into one
shared library next to this file.  quantize.cu is compiled without FMA
contraction so the quantizer's f32 arithmetic rounds exactly where the
page's does.

build(debug=True) makes libq4_debug.so from the same sources with
-DQ4_DEBUG: every global store of the kernels is checked against its
buffer's extent, and one outside it is recorded in the device error word
(q4_check then returns Q4_ERR_BOUNDS) and skipped.  The package loads it
when Q4_LIBRARY names it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libq4.so")
LIB_DEBUG = os.path.join(HERE, "libq4_debug.so")
BUILD = os.path.join(ROOT, "_build", "q4")
BUILD_DEBUG = os.path.join(ROOT, "_build", "q4_debug")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
SOURCES = {
    "api.cu": [],
    "quantize.cu": ["--fmad=false", "-prec-div=true", "-ftz=false"],
    "gemv.cu": [],
    "gemm_tc.cu": [],
    "noalloc.cu": [],
}


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return p


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src, os.path.join(CSRC, "common.cuh"), os.path.join(ROOT, "include", "q4.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra: list | None = None,
          debug: bool = False) -> str:
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    extra = (["-DQ4_DEBUG"] if debug else []) + list(extra or [])
    os.makedirs(build_dir, exist_ok=True)
    # objects built on another machine type are never reused
    stamp = os.path.join(build_dir, "machine")
    machine = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != machine:
        force = True
        with open(stamp, "w") as f:
            f.write(machine)
    jobs = []
    for name, flags in SOURCES.items():
        src = os.path.join(CSRC, name)
        obj = os.path.join(build_dir, name + ".o")
        if force or _stale(obj, src):
            cmd = [nvcc(), *ARCH, *COMMON, *flags, *extra, "-c", src, "-o", obj]
            jobs.append(cmd)
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(subprocess.run, c, capture_output=True, text=True) for c in jobs]
            for c, f in zip(jobs, futs):
                r = f.result()
                if verbose or r.returncode:
                    print(" ".join(c))
                    print(r.stdout, r.stderr)
                if r.returncode:
                    raise RuntimeError(f"nvcc failed for {c[-3]}")
    objs = [os.path.join(build_dir, n + ".o") for n in SOURCES]
    if jobs or force or not os.path.exists(lib):
        cmd = [nvcc(), *ARCH, "-shared", "-o", lib, *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            print(r.stdout, r.stderr)
            raise RuntimeError(f"link of {os.path.basename(lib)} failed")
    return lib


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
