"""Build libq4.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu file is compiled to an object in parallel, then linked into one
shared library next to this file.  quantize.cu is compiled without FMA
contraction so the quantizer's f32 arithmetic rounds exactly where the
page's does.
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
BUILD = os.path.join(ROOT, "_build", "q4")
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


def build(verbose: bool = False, force: bool = False, extra: list | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    # objects built on another machine type are never reused
    stamp = os.path.join(BUILD, "machine")
    machine = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != machine:
        force = True
        with open(stamp, "w") as f:
            f.write(machine)
    jobs = []
    for name, flags in SOURCES.items():
        src = os.path.join(CSRC, name)
        obj = os.path.join(BUILD, name + ".o")
        if force or _stale(obj, src):
            cmd = [nvcc(), *ARCH, *COMMON, *flags, *(extra or []), "-c", src, "-o", obj]
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
    objs = [os.path.join(BUILD, n + ".o") for n in SOURCES]
    if jobs or force or not os.path.exists(LIB):
        cmd = [nvcc(), *ARCH, "-shared", "-o", LIB, *objs, "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            print(r.stdout, r.stderr)
            raise RuntimeError("link of libq4.so failed")
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
