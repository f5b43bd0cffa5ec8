"""Python binding of libq4.so, the GB300 weight-only INT4 group-128 library.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch is used for device memory and the current CUDA stream.  Importing
this package fails loudly when libq4.so has not been built; there is no
fallback of any kind.

Names follow include/q4.h: quantize, quantize_sym, repack, unpack, xsum,
gemv, gemm, check, weight_bytes, gemv_workspace_bytes, gemm_workspace_bytes,
repack_compact, unpack_compact, gemv_noalloc and the two timeout
self-tests.  A QWeight carries its layout (TILED or COMPACT), and every
product call passes that layout and the buffer's byte count to the library,
which refuses a mismatch.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# Q4_LIBRARY selects another build of the same library (the bounds-checked
# libq4_debug.so); the named file must exist, there is no fallback.
LIB_PATH = os.environ.get("Q4_LIBRARY") or os.path.join(_HERE, "libq4.so")
GROUP = 128
TILE_ROWS = 16
TILE_BYTES = 1104
CMP_TILE_BYTES = 1072
GEMV_MAX_M = 16

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = range(7)
F32, BF16, F16 = 0, 1, 2
LAYOUT_TILED, LAYOUT_COMPACT = 1, 2
PATH_AUTO, PATH_FMA, PATH_MMA = 0, 1, 2

_DTYPE = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.q4_status_str(status).decode()
        if status == ERR_CUDA:
            msg += ": " + _lib.q4_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, Z, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    lib.q4_quantize.argtypes = [P, I, I, P, P, P, P]
    lib.q4_quantize_sym.argtypes = [P, I, I, P, P, P, P]
    lib.q4_weight_bytes.argtypes = [I, I, S]
    lib.q4_weight_bytes.restype = Z
    lib.q4_repack.argtypes = [P, P, P, I, I, P, P]
    lib.q4_unpack.argtypes = [P, I, I, P, P, P, P]
    lib.q4_repack_compact.argtypes = [P, P, P, I, I, P, P]
    lib.q4_unpack_compact.argtypes = [P, I, I, P, P, P, P]
    lib.q4_xsum.argtypes = [P, S, I, I, P, P]
    lib.q4_gemv_workspace_bytes.argtypes = [I, I, I]
    lib.q4_gemv_workspace_bytes.restype = Z
    lib.q4_gemm_workspace_bytes.argtypes = [I, I, I]
    lib.q4_gemm_workspace_bytes.restype = Z
    prod = [P, S, I, I, I, P, S, Z, P, S, P, Z, P]  # x, xt, M, N, K, qw, layout, bytes, y, yt, ws, wsb, stream
    lib.q4_gemv.argtypes = prod
    lib.q4_gemv_path.argtypes = prod[:-1] + [S, P]
    lib.q4_gemv_timeout_selftest.argtypes = prod
    lib.q4_gemm.argtypes = prod
    lib.q4_gemm_timeout_selftest.argtypes = prod
    lib.q4_gemv_noalloc.argtypes = [P, S, I, I, I, P, S, Z, P, S, P]
    lib.q4_check.argtypes = [P]
    lib.q4_debug_bounds_selftest.argtypes = [P, P]
    lib.q4_status_str.argtypes = [S]
    lib.q4_status_str.restype = ctypes.c_char_p
    lib.q4_last_cuda_error.restype = ctypes.c_char_p
    for f in ("q4_quantize", "q4_quantize_sym", "q4_repack", "q4_unpack", "q4_repack_compact",
              "q4_unpack_compact", "q4_xsum", "q4_gemv", "q4_gemv_path", "q4_gemv_timeout_selftest",
              "q4_gemm", "q4_gemm_timeout_selftest", "q4_gemv_noalloc", "q4_check",
              "q4_debug_bounds_selftest"):
        getattr(lib, f).restype = S
    return lib


_lib = _load()


def lib():
    """The loaded ctypes library (for callers that marshal their own pointers)."""
    return _lib


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ok(status: int, where: str):
    if status != OK:
        raise Q4Error(status, where)


def _cuda(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ API
def weight_bytes(N: int, K: int, layout: int = LAYOUT_TILED) -> int:
    return int(_lib.q4_weight_bytes(N, K, layout))


def weight_bytes_compact(N: int, K: int) -> int:
    return weight_bytes(N, K, LAYOUT_COMPACT)


def gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.q4_gemv_workspace_bytes(M, N, K))


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.q4_gemm_workspace_bytes(M, N, K))


def quantize(w: torch.Tensor, stream=None, symmetric: bool = False):
    """w f32 [N][K] (cuda) -> (packed u8 [N][K/2], scale f32 [N][K/128], zero u8 [N][K/128]).

    ``symmetric`` calls q4_quantize_sym (max|w|/7 scales, zero 8)."""
    _cuda(w, "w")
    if w.dtype != torch.float32 or w.dim() != 2:
        raise ValueError("w must be a 2-D float32 tensor")
    N, K = w.shape
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device)
    scale = torch.empty((N, max(K // GROUP, 1)), dtype=torch.float32, device=w.device)
    zero = torch.empty((N, max(K // GROUP, 1)), dtype=torch.uint8, device=w.device)
    fn, name = (_lib.q4_quantize_sym, "q4_quantize_sym") if symmetric else \
        (_lib.q4_quantize, "q4_quantize")
    _ok(fn(w.data_ptr(), N, K, packed.data_ptr(), scale.data_ptr(), zero.data_ptr(),
           _stream(stream)), name)
    return packed, scale, zero


def quantize_sym(w: torch.Tensor, stream=None):
    """Symmetric group-128 quantization (q4_quantize_sym); same outputs as quantize."""
    return quantize(w, stream, symmetric=True)


def repack(packed: torch.Tensor, scale: torch.Tensor, zero: torch.Tensor, N: int, K: int,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical arrays -> tiled kernel layout (uint8 [weight_bytes(N, K)])."""
    for t, n in ((packed, "packed"), (scale, "scale"), (zero, "zero")):
        _cuda(t, n)
    nb = weight_bytes(N, K)
    if nb == 0:
        raise ValueError(f"invalid shape {N}x{K}")
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=packed.device)
    _ok(_lib.q4_repack(packed.data_ptr(), scale.data_ptr(), zero.data_ptr(), N, K,
                       out.data_ptr(), _stream(stream)), "q4_repack")
    return out


def unpack(qw: torch.Tensor, N: int, K: int, stream=None):
    _cuda(qw, "qw")
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=qw.device)
    scale = torch.empty((N, K // GROUP), dtype=torch.float32, device=qw.device)
    zero = torch.empty((N, K // GROUP), dtype=torch.uint8, device=qw.device)
    _ok(_lib.q4_unpack(qw.data_ptr(), N, K, packed.data_ptr(), scale.data_ptr(),
                       zero.data_ptr(), _stream(stream)), "q4_unpack")
    return packed, scale, zero


def repack_compact(packed: torch.Tensor, scale: torch.Tensor, zero: torch.Tensor, N: int, K: int,
                   out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical arrays -> compact tiles (binary16 scales, 4-bit zeros)."""
    for t, n in ((packed, "packed"), (scale, "scale"), (zero, "zero")):
        _cuda(t, n)
    nb = weight_bytes(N, K, LAYOUT_COMPACT)
    if nb == 0:
        raise ValueError(f"invalid shape {N}x{K}")
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=packed.device)
    _ok(_lib.q4_repack_compact(packed.data_ptr(), scale.data_ptr(), zero.data_ptr(), N, K,
                               out.data_ptr(), _stream(stream)), "q4_repack_compact")
    return out


def unpack_compact(qw: torch.Tensor, N: int, K: int, stream=None):
    """Compact tiles -> (codes u8 [N][K/2], binary16 scale bits int16 [N][K/128], zeros u8 [N][K/128])."""
    _cuda(qw, "qw")
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=qw.device)
    scale16 = torch.empty((N, K // GROUP), dtype=torch.int16, device=qw.device)
    zero = torch.empty((N, K // GROUP), dtype=torch.uint8, device=qw.device)
    _ok(_lib.q4_unpack_compact(qw.data_ptr(), N, K, packed.data_ptr(), scale16.data_ptr(),
                               zero.data_ptr(), _stream(stream)), "q4_unpack_compact")
    return packed, scale16, zero


def xsum(x: torch.Tensor, stream=None) -> torch.Tensor:
    _cuda(x, "x")
    M, K = x.shape
    out = torch.empty((M, K // GROUP), dtype=torch.float32, device=x.device)
    _ok(_lib.q4_xsum(x.data_ptr(), _DTYPE[x.dtype], M, K, out.data_ptr(), _stream(stream)),
        "q4_xsum")
    return out


@dataclass
class QWeight:
    """A weight matrix in one of the tiled kernel layouts (compact: binary16
    scales and 4-bit zeros)."""
    data: torch.Tensor  # uint8 [weight_bytes(N, K, layout)]
    N: int
    K: int
    compact: bool = False

    @property
    def layout(self) -> int:
        return LAYOUT_COMPACT if self.compact else LAYOUT_TILED

    @property
    def nbytes(self) -> int:
        return self.data.numel() * self.data.element_size()

    @classmethod
    def from_float(cls, w: torch.Tensor, stream=None, symmetric: bool = False,
                   compact: bool = False) -> "QWeight":
        N, K = w.shape
        packed, scale, zero = quantize(w, stream, symmetric=symmetric)
        if compact:
            return cls(repack_compact(packed, scale, zero, N, K, stream=stream), N, K, True)
        return cls(repack(packed, scale, zero, N, K, stream=stream), N, K)


def _zeros(nb: int, device) -> torch.Tensor | None:
    if nb == 0:
        return None
    return torch.zeros(nb, dtype=torch.uint8, device=device or torch.cuda.current_device())


def workspace(M: int, N: int, K: int, device=None) -> torch.Tensor | None:
    """A zero-filled workspace for q4_gemv (None when none is needed)."""
    return _zeros(gemv_workspace_bytes(M, N, K), device)


def gemm_workspace(M: int, N: int, K: int, device=None) -> torch.Tensor | None:
    """A zero-filled workspace for q4_gemm (None when none is needed)."""
    return _zeros(gemm_workspace_bytes(M, N, K), device)


def _ws(ws):
    return (0, 0) if ws is None else (ws.data_ptr(), ws.numel())


def _product_args(x: torch.Tensor, qw: QWeight, out_dtype, out):
    _cuda(x, "x")
    M, K = x.shape
    if K != qw.K:
        raise ValueError(f"x has K={K}, weight has K={qw.K}")
    if out is None:
        out = torch.empty((M, qw.N), dtype=out_dtype or x.dtype, device=x.device)
    return M, K, out


def gemv(x: torch.Tensor, qw: QWeight, out_dtype=None, out: torch.Tensor | None = None,
         ws: torch.Tensor | None = None, path: int = PATH_AUTO, stream=None) -> torch.Tensor:
    """y [M][N] = x [M][K] * w_hat^T for 1 <= M <= 16."""
    M, K, out = _product_args(x, qw, out_dtype, out)
    if ws is None:
        ws = workspace(M, qw.N, K, x.device)
    wsp, wsb = _ws(ws)
    _ok(_lib.q4_gemv_path(x.data_ptr(), _DTYPE[x.dtype], M, qw.N, K, qw.data.data_ptr(),
                          qw.layout, qw.nbytes, out.data_ptr(), _DTYPE[out.dtype], wsp, wsb,
                          path, _stream(stream)), "q4_gemv")
    return out


def gemv_noalloc(x: torch.Tensor, qw: QWeight, out_dtype=None, out: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """q4_gemv_noalloc: q4_gemv with the library's static scratch array as
    its workspace (for callers that cannot allocate device memory)."""
    M, K, out = _product_args(x, qw, out_dtype, out)
    _ok(_lib.q4_gemv_noalloc(x.data_ptr(), _DTYPE[x.dtype], M, qw.N, K, qw.data.data_ptr(),
                             qw.layout, qw.nbytes, out.data_ptr(), _DTYPE[out.dtype],
                             _stream(stream)), "q4_gemv_noalloc")
    return out


def gemv_timeout_selftest(x: torch.Tensor, qw: QWeight, out: torch.Tensor,
                          ws: torch.Tensor | None = None, stream=None) -> None:
    M, K = x.shape
    wsp, wsb = _ws(ws)
    _ok(_lib.q4_gemv_timeout_selftest(x.data_ptr(), _DTYPE[x.dtype], M, qw.N, K,
                                      qw.data.data_ptr(), qw.layout, qw.nbytes, out.data_ptr(),
                                      _DTYPE[out.dtype], wsp, wsb, _stream(stream)),
        "q4_gemv_timeout_selftest")


def gemm(x: torch.Tensor, qw: QWeight, out_dtype=None, out: torch.Tensor | None = None,
         ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y [M][N] = X [M][K] * w_hat^T on the tcgen05 tensor cores (any M)."""
    M, K, out = _product_args(x, qw, out_dtype, out)
    if ws is None:
        ws = gemm_workspace(M, qw.N, K, x.device)
    wsp, wsb = _ws(ws)
    _ok(_lib.q4_gemm(x.data_ptr(), _DTYPE[x.dtype], M, qw.N, K, qw.data.data_ptr(), qw.layout,
                     qw.nbytes, out.data_ptr(), _DTYPE[out.dtype], wsp, wsb, _stream(stream)),
        "q4_gemm")
    return out


def gemm_timeout_selftest(x: torch.Tensor, qw: QWeight, out: torch.Tensor,
                          ws: torch.Tensor | None = None, stream=None) -> None:
    M, K = x.shape
    wsp, wsb = _ws(ws)
    _ok(_lib.q4_gemm_timeout_selftest(x.data_ptr(), _DTYPE[x.dtype], M, qw.N, K,
                                      qw.data.data_ptr(), qw.layout, qw.nbytes, out.data_ptr(),
                                      _DTYPE[out.dtype], wsp, wsb, _stream(stream)),
        "q4_gemm_timeout_selftest")


def check(stream=None) -> int:
    """Synchronise and return the library status (raises nothing)."""
    return int(_lib.q4_check(_stream(stream)))
