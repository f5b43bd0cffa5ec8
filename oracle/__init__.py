"""CPU oracle for group-128 INT4 quantization (asymmetric and symmetric) and the
W4A16 product.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product library never imports it,
and it never imports the product library.

The arithmetic lives in plain C (``oq4.c``), written from the page "Weight
quantization" (tirogla.com), sections "How it works" and "Code"; the
symmetric scheme from the page "Quantization" (hritesh-sonawane.github.io
notes), sections "How it really works" and "Code".  This module
only compiles it with gcc and marshals numpy arrays through ctypes.  ctypes
releases the GIL during each call, so callers may run disjoint row ranges on
several Python threads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oq4.c")
_LIB = os.path.join(_HERE, "liboq4.so")
G = 128

_CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(out: str = _LIB, mutant: int = 0, quiet: bool = True) -> str:
    """Compile oq4.c into a shared library (``mutant`` > 0 plants a known bug)."""
    cmd = ["gcc", *_CFLAGS, f"-DOQ4_MUTANT={int(mutant)}", "-o", out, _SRC, "-lm"]
    subprocess.run(cmd, check=True, capture_output=quiet)
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(os.path.join(_HERE, f)) > t for f in ("oq4.c", "oq4.h"))


_P = ctypes.c_void_p
_I = ctypes.c_int64


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        lib.oq4_quantize_g.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        lib.oq4_quantize_g.restype = ctypes.c_int
        lib.oq4_quantize_sym_g.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        lib.oq4_quantize_sym_g.restype = ctypes.c_int
        lib.oq4_dequant_g.argtypes = [_P, _P, _P, _I, _I, _I, _P]
        lib.oq4_dequant_g.restype = None
        lib.oq4_dot_naive.argtypes = [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P, _P]
        lib.oq4_dot_naive.restype = None
        lib.oq4_dot_factored.argtypes = [_P, _I, _P, _P, _P, _I, _I, _I, _I, _P]
        lib.oq4_dot_factored.restype = None
        lib.oq4_xsum.argtypes = [_P, _I, _I, _P]
        lib.oq4_xsum.restype = None
        lib.oq4_f16_bits.argtypes = [ctypes.c_float]
        lib.oq4_f16_bits.restype = ctypes.c_uint16
        lib.oq4_f16_value.argtypes = [ctypes.c_uint16]
        lib.oq4_f16_value.restype = ctypes.c_float
        lib.oq4_compact_meta.argtypes = [_P, _P, _I, _I, _P, _P]
        lib.oq4_compact_meta.restype = None
        lib.oq4_expand_meta.argtypes = [_P, _P, _I, _I, _P, _P]
        lib.oq4_expand_meta.restype = None
        lib.oq4_mutant.restype = ctypes.c_int
        self.lib = lib
        self.path = path
        self.mutant = lib.oq4_mutant()

    # -- quantize / dequantize ------------------------------------------------
    def quantize(self, w: np.ndarray, group: int = G, symmetric: bool = False):
        """w: f32 [N][K] -> (packed u8 [N][K/2], scale f32 [N][K/G], zero u8 [N][K/G]).

        ``symmetric`` selects the absmax/7 scheme (codes q + 8, zero 8)."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        if w.ndim == 1:
            w = w[None, :]
        N, K = w.shape
        packed = np.zeros((N, K // 2), np.uint8)
        scale = np.zeros((N, K // group), np.float32)
        zero = np.zeros((N, K // group), np.uint8)
        fn = self.lib.oq4_quantize_sym_g if symmetric else self.lib.oq4_quantize_g
        rc = fn(w.ctypes.data, N, K, group, packed.ctypes.data, scale.ctypes.data,
                zero.ctypes.data)
        if rc != 0:
            raise ValueError(f"oracle quantize rejected shape {N}x{K} with G={group}")
        return packed, scale, zero

    # -- compact metadata (binary16 scales, 4-bit zeros) ---------------------
    def f16_bits(self, v: np.ndarray) -> np.ndarray:
        v = np.ascontiguousarray(v, np.float32).reshape(-1)
        return np.array([self.lib.oq4_f16_bits(float(x)) for x in v], np.uint16)

    def f16_values(self, h: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(h, np.uint16).reshape(-1)
        return np.array([self.lib.oq4_f16_value(int(x)) for x in h], np.float32)

    def compact_meta(self, scale, zero):
        """scale f32 [N][NG], zero u8 [N][NG] -> (scale16 u16 [N][NG], zero4 u8 [N][ceil(NG/2)])."""
        scale = np.ascontiguousarray(scale, np.float32)
        zero = np.ascontiguousarray(zero, np.uint8)
        N, NG = scale.shape
        s16 = np.empty((N, NG), np.uint16)
        z4 = np.empty((N, (NG + 1) // 2), np.uint8)
        self.lib.oq4_compact_meta(scale.ctypes.data, zero.ctypes.data, N, NG, s16.ctypes.data,
                                  z4.ctypes.data)
        return s16, z4

    def expand_meta(self, scale16, zero4, NG: int):
        """Inverse containers: (scale f32 [N][NG] widened from binary16, zero u8 [N][NG])."""
        scale16 = np.ascontiguousarray(scale16, np.uint16)
        zero4 = np.ascontiguousarray(zero4, np.uint8)
        N = scale16.shape[0]
        scale = np.empty((N, NG), np.float32)
        zero = np.empty((N, NG), np.uint8)
        self.lib.oq4_expand_meta(scale16.ctypes.data, zero4.ctypes.data, N, NG, scale.ctypes.data,
                                 zero.ctypes.data)
        return scale, zero

    def dequant(self, packed, scale, zero, N: int, K: int, group: int = G) -> np.ndarray:
        packed = np.ascontiguousarray(packed, np.uint8)
        scale = np.ascontiguousarray(scale, np.float32)
        zero = np.ascontiguousarray(zero, np.uint8)
        out = np.empty((N, K), np.float64)
        self.lib.oq4_dequant_g(packed.ctypes.data, scale.ctypes.data, zero.ctypes.data,
                               N, K, group, out.ctypes.data)
        return out

    # -- products -------------------------------------------------------------
    def dot_naive(self, x, packed, scale, zero, N: int, K: int, n0: int = 0, n1=None,
                  threads: int = 1):
        """Definition in double. Returns (y [M][n1-n0], absdot [M][n1-n0])."""
        n1 = N if n1 is None else n1
        x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
        packed = np.ascontiguousarray(packed, np.uint8)
        scale = np.ascontiguousarray(scale, np.float32)
        zero = np.ascontiguousarray(zero, np.uint8)
        M = x.shape[0]
        y = np.empty((M, n1 - n0), np.float64)
        a = np.empty((M, n1 - n0), np.float64)

        def run(lo, hi):
            ys = np.empty((M, hi - lo), np.float64)
            as_ = np.empty((M, hi - lo), np.float64)
            self.lib.oq4_dot_naive(x.ctypes.data, M, packed.ctypes.data, scale.ctypes.data,
                                   zero.ctypes.data, N, K, lo, hi, ys.ctypes.data,
                                   as_.ctypes.data)
            y[:, lo - n0:hi - n0] = ys
            a[:, lo - n0:hi - n0] = as_

        _split(run, n0, n1, threads)
        return y, a

    def dot_factored(self, x, packed, scale, zero, N: int, K: int, n0: int = 0, n1=None,
                     threads: int = 1):
        """The page's factored dot in f32. Returns y f32 [M][n1-n0]."""
        n1 = N if n1 is None else n1
        x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
        packed = np.ascontiguousarray(packed, np.uint8)
        scale = np.ascontiguousarray(scale, np.float32)
        zero = np.ascontiguousarray(zero, np.uint8)
        M = x.shape[0]
        y = np.empty((M, n1 - n0), np.float32)

        def run(lo, hi):
            ys = np.empty((M, hi - lo), np.float32)
            self.lib.oq4_dot_factored(x.ctypes.data, M, packed.ctypes.data, scale.ctypes.data,
                                      zero.ctypes.data, N, K, lo, hi, ys.ctypes.data)
            y[:, lo - n0:hi - n0] = ys

        _split(run, n0, n1, threads)
        return y

    def xsum(self, x) -> np.ndarray:
        x = np.ascontiguousarray(np.atleast_2d(x), np.float32)
        M, K = x.shape
        out = np.empty((M, K // G), np.float64)
        self.lib.oq4_xsum(x.ctypes.data, M, K, out.ctypes.data)
        return out


def _split(run, n0: int, n1: int, threads: int) -> None:
    threads = max(1, min(threads, n1 - n0))
    if threads == 1:
        run(n0, n1)
        return
    bounds = np.linspace(n0, n1, threads + 1).astype(np.int64)
    ts = [threading.Thread(target=run, args=(int(bounds[i]), int(bounds[i + 1])))
          for i in range(threads) if bounds[i + 1] > bounds[i]]
    for t in ts:
        t.start()
    for t in ts:
        t.join()


_default = None
_lock = threading.Lock()


def load() -> Oracle:
    """The real oracle (mutant 0), compiled on first use if missing or stale."""
    global _default
    with _lock:
        if _default is None:
            if _stale(_LIB):
                build(_LIB)
            _default = Oracle(_LIB)
    return _default


def load_mutant(mutant: int, workdir: str) -> Oracle:
    """Compile and load the oracle with planted mistake number ``mutant``."""
    path = os.path.join(workdir, f"liboq4_m{mutant}.so")
    build(path, mutant=mutant)
    return Oracle(path)
