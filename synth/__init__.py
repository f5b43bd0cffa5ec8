"""Seeded synthetic inputs shared by the oracle side and the GPU side.

Holds no quantization or matmul arithmetic: only random draws and dtype
rounding (see ``synth.h`` for the generator definitions).  Host draws come
from ``libq4synth.so`` (gcc); device draws come from ``libq4synth_dev.so``
(nvcc), bit-identical to the host ones.

Workload recipes (shapes and distributions of the pages' workloads):
  * ``page_program``: the n=4096 experiment of the page "Weight quantization",
    section "Code" (xorshift stream; w = 0.02*U(-1,1) first, then x = U(-1,1)).
  * ``xorshift_matrix``: the same stream drawn for an N x K weight matrix
    (row-major) followed by K activations -- the 4096x4096 single-GEMV case.
  * ``normal_rows`` / ``dev_normal_f32``: W ~ N(0, sigma) per element by flat
    index, optional outlier columns multiplied by a factor.
  * ``normal_bf16`` / ``dev_normal_bf16``: activations ~ N(0,1) rounded to bf16.
  * ``row_scaled_outliers``: the 256x1024 matrix with per-row spreads and
    eight outliers of the page "Quantization" (hritesh-sonawane.github.io
    notes), section "Code" (Python's Mersenne Twister).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_LIB = os.path.join(_HERE, "libq4synth.so")
_DEV_LIB = os.path.join(_HERE, "libq4synth_dev.so")
PAGE_SEED = 0x9E3779B97F4A7C15

_P = ctypes.c_void_p
_I = ctypes.c_int64
_U = ctypes.c_uint64
_F = ctypes.c_float


def build_host(quiet: bool = True) -> str:
    src = os.path.join(_HERE, "synth.c")
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared", "-o", _HOST_LIB, src]
    subprocess.run(cmd, check=True, capture_output=quiet)
    return _HOST_LIB


def build_dev_cmd() -> list:
    src = os.path.join(_HERE, "synth_dev.cu")
    return ["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
            "--fmad=false", "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_LIB, src]


def build_dev(quiet: bool = True) -> str:
    subprocess.run(build_dev_cmd(), check=True, capture_output=quiet)
    return _DEV_LIB


def _stale(lib, srcs):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(os.path.join(_HERE, s)) > t for s in srcs)


_host = None
_dev = None


def host():
    global _host
    if _host is None:
        if _stale(_HOST_LIB, ("synth.c", "synth.h")):
            build_host()
        lib = ctypes.CDLL(_HOST_LIB)
        lib.synth_xorshift_f32.argtypes = [ctypes.POINTER(_U), _I, _P]
        lib.synth_uniform_f32.argtypes = [_U, _I, _I, _F, _P]
        lib.synth_normal_f32.argtypes = [_U, _I, _I, _F, _P]
        lib.synth_normal_rows_f32.argtypes = [_U, _I, _I, _I, _F, _P, _I, _F, _P]
        lib.synth_f32_to_bf16.argtypes = [_P, _I, _P]
        lib.synth_sample_without_replacement.argtypes = [_U, _I, _I, _P]
        for f in ("synth_xorshift_f32", "synth_uniform_f32", "synth_normal_f32",
                  "synth_normal_rows_f32", "synth_f32_to_bf16",
                  "synth_sample_without_replacement"):
            getattr(lib, f).restype = None
        _host = lib
    return _host


def dev():
    global _dev
    if _dev is None:
        if _stale(_DEV_LIB, ("synth_dev.cu",)):
            build_dev()
        lib = ctypes.CDLL(_DEV_LIB)
        lib.synth_dev_normal_f32.argtypes = [_P, _I, _U, _I, _F, _P, _I, _F, _P]
        lib.synth_dev_uniform_f32.argtypes = [_P, _I, _U, _I, _F, _P]
        lib.synth_dev_normal_bf16.argtypes = [_P, _I, _U, _I, _F, _P]
        for f in ("synth_dev_normal_f32", "synth_dev_uniform_f32", "synth_dev_normal_bf16"):
            getattr(lib, f).restype = ctypes.c_int
        _dev = lib
    return _dev


# --------------------------------------------------------------------------- host
def xorshift_stream(count: int, state: int = PAGE_SEED):
    """The page's xorshift draws in [-1, 1). Returns (values f32, new_state)."""
    st = _U(state)
    out = np.empty(count, np.float32)
    host().synth_xorshift_f32(ctypes.byref(st), count, out.ctypes.data)
    return out, st.value


def page_program(n: int = 4096):
    """(w, x) of the page's experiment: w = 0.02*rnd() for n draws, then x = rnd()."""
    r, _ = xorshift_stream(2 * n)
    w = (np.float32(0.02) * r[:n]).astype(np.float32)
    x = r[n:].copy()
    return w, x


def xorshift_matrix(N: int, K: int):
    """W f32 [N][K] = 0.02*rnd() row-major, then x f32 [K] = rnd(), one stream."""
    r, _ = xorshift_stream(N * K + K)
    W = (np.float32(0.02) * r[:N * K]).astype(np.float32).reshape(N, K)
    return W, r[N * K:].copy()


def row_scaled_outliers(rows: int = 256, cols: int = 1024, seed: int = 11,
                        n_outliers: int = 8, magnitude: float = 0.6) -> np.ndarray:
    """The synthetic matrix of the page "Quantization" (hritesh-sonawane.github.io
    notes), section "Code": each row draws its own spread 0.02*exp(N(0, 0.5))
    and then ``cols`` values N(0, spread); afterwards ``n_outliers`` entries
    become +-``magnitude``, each drawing its sign, then its row, then its
    column.  Draws come from Python's own generator (``random.Random``,
    Mersenne Twister, its ``gauss``) in exactly that order, so the error table
    the page prints for this matrix applies to it.  Returns f64 [rows][cols]."""
    import math
    import random

    gen = random.Random(seed)
    out = np.empty((rows, cols), np.float64)
    for r in range(rows):
        spread = 0.02 * math.exp(gen.gauss(0.0, 0.5))
        out[r, :] = [gen.gauss(0.0, spread) for _c in range(cols)]
    for _i in range(n_outliers):
        sign = gen.choice((-1, 1))
        r = gen.randrange(rows)
        c = gen.randrange(cols)
        out[r, c] = sign * magnitude
    return out


def uniform(seed: int, start: int, count: int, scale: float = 1.0) -> np.ndarray:
    out = np.empty(count, np.float32)
    host().synth_uniform_f32(seed, start, count, scale, out.ctypes.data)
    return out


def normal(seed: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    out = np.empty(count, np.float32)
    host().synth_normal_f32(seed, start, count, sigma, out.ctypes.data)
    return out


def normal_rows(seed: int, C: int, r0: int, r1: int, sigma: float, cols=None,
                factor: float = 1.0) -> np.ndarray:
    """Rows [r0, r1) of the matrix with element (r, c) = sigma*normal(r*C + c)."""
    cols = np.zeros(0, np.int32) if cols is None else np.ascontiguousarray(cols, np.int32)
    out = np.empty((r1 - r0, C), np.float32)
    host().synth_normal_rows_f32(seed, C, r0, r1, sigma, cols.ctypes.data, len(cols), factor,
                                 out.ctypes.data)
    return out


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, np.float32)
    out = np.empty(a.shape, np.uint16)
    host().synth_f32_to_bf16(a.ctypes.data, a.size, out.ctypes.data)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, start: int, count: int, sigma: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of sigma*normal(start + j)."""
    return to_bf16_bits(normal(seed, start, count, sigma))


def outlier_columns(seed: int, K: int, frac: float = 0.001) -> np.ndarray:
    """round(frac*K) distinct input channels, sorted (seeded sampling)."""
    count = int(round(frac * K))
    out = np.empty(count, np.int32)
    if count:
        host().synth_sample_without_replacement(seed, K, count, out.ctypes.data)
    return out


# --------------------------------------------------------------------------- device
def _stream_ptr(stream):
    return ctypes.c_void_p(0 if stream is None else stream)


def dev_normal_f32(ptr: int, count: int, seed: int, start: int = 0, sigma: float = 1.0,
                   col_mask_ptr: int = 0, C: int = 1, factor: float = 1.0, stream=None):
    rc = dev().synth_dev_normal_f32(ptr, count, seed, start, sigma, col_mask_ptr or None, C,
                                    factor, _stream_ptr(stream))
    if rc:
        raise RuntimeError(f"synth_dev_normal_f32 failed: cuda error {rc}")


def dev_uniform_f32(ptr: int, count: int, seed: int, start: int = 0, scale: float = 1.0,
                    stream=None):
    rc = dev().synth_dev_uniform_f32(ptr, count, seed, start, scale, _stream_ptr(stream))
    if rc:
        raise RuntimeError(f"synth_dev_uniform_f32 failed: cuda error {rc}")


def dev_normal_bf16(ptr: int, count: int, seed: int, start: int = 0, sigma: float = 1.0,
                    stream=None):
    rc = dev().synth_dev_normal_bf16(ptr, count, seed, start, sigma, _stream_ptr(stream))
    if rc:
        raise RuntimeError(f"synth_dev_normal_bf16 failed: cuda error {rc}")
