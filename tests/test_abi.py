"""The C-ABI library: loads, exports every symbol include/q4.h declares, and
rejects bad arguments on the host before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4.h")
LIB = os.path.join(ROOT, "weight_only_int4_group_gb300", "libq4.so")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("q4_quantize", "q4_quantize_sym", "q4_repack", "q4_unpack", "q4_repack_compact",
                 "q4_unpack_compact", "q4_xsum", "q4_gemv", "q4_gemv_path", "q4_gemm",
                 "q4_check", "q4_status_str", "q4_weight_bytes", "q4_gemv_workspace_bytes",
                 "q4_gemm_workspace_bytes", "q4_gemv_timeout_selftest", "q4_gemm_timeout_selftest",
                 "q4_gemv_noalloc", "q4_debug_bounds_selftest"):
        assert must in names


def test_header_is_plain_c():
    text = open(HEADER).read()
    assert "torch" not in text.lower().replace("pytorch", "")
    assert "#include <cuda" not in text


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in q4.h but not exported"


def test_status_strings(lib):
    lib.q4_status_str.restype = ctypes.c_char_p
    for s in range(7):
        assert lib.q4_status_str(s)
    assert b"unknown" in lib.q4_status_str(99)


TILED, COMPACT = 1, 2


def test_weight_bytes(lib):
    lib.q4_weight_bytes.restype = ctypes.c_size_t
    lib.q4_weight_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int]
    assert lib.q4_weight_bytes(16, 128, TILED) == 1104
    assert lib.q4_weight_bytes(17, 256, TILED) == 2 * 2 * 1104
    assert lib.q4_weight_bytes(28672, 8192, TILED) == 1792 * 64 * 1104
    assert lib.q4_weight_bytes(17, 256, COMPACT) == 2 * 2 * 1072
    assert lib.q4_weight_bytes(16, 100, TILED) == 0
    assert lib.q4_weight_bytes(0, 128, TILED) == 0
    assert lib.q4_weight_bytes(16, 128, 0) == 0  # unknown layout
    assert lib.q4_weight_bytes(16, 128, 3) == 0


def _product_argtypes(lib):
    P, I, S, Z = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    prod = [P, S, I, I, I, P, S, Z, P, S, P, Z, P]
    for f in ("q4_gemv", "q4_gemm", "q4_gemv_timeout_selftest", "q4_gemm_timeout_selftest"):
        getattr(lib, f).argtypes = prod
        getattr(lib, f).restype = S
    lib.q4_gemv_path.argtypes = prod[:-1] + [S, P]
    lib.q4_gemv_noalloc.argtypes = [P, S, I, I, I, P, S, Z, P, S, P]


def test_host_side_argument_errors(lib):
    P, I, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.q4_quantize.argtypes = [P, I, I, P, P, P, P]
    lib.q4_repack.argtypes = [P, P, P, I, I, P, P]
    _product_argtypes(lib)
    fake = 4096  # never dereferenced: every case below fails its host checks first
    # NULL pointer, bad K, K not a multiple of 128
    assert lib.q4_quantize(None, 4, 128, fake, fake, fake, None) == 1
    assert lib.q4_quantize(fake, 4, 100, fake, fake, fake, None) == 1
    assert lib.q4_quantize(fake, 0, 128, fake, fake, fake, None) == 1
    # misaligned input
    assert lib.q4_quantize(fake + 4, 4, 128, fake, fake, fake, None) == 3
    # compact tiles: the same checks as the canonical layout
    lib.q4_repack_compact.argtypes = [P, P, P, I, I, P, P]
    assert lib.q4_repack_compact(fake, fake, fake, 4, 128, fake + 8, None) == 3
    assert lib.q4_repack_compact(fake, fake, fake, 4, 100, fake, None) == 1
    # the symmetric quantizer shares the checks
    lib.q4_quantize_sym.argtypes = [P, I, I, P, P, P, P]
    assert lib.q4_quantize_sym(None, 4, 128, fake, fake, fake, None) == 1
    assert lib.q4_quantize_sym(fake, 4, 100, fake, fake, fake, None) == 1
    assert lib.q4_quantize_sym(fake + 4, 4, 128, fake, fake, fake, None) == 3
    assert lib.q4_repack(fake, fake, fake, 4, 128, fake + 8, None) == 3
    wb = 4 * 1104  # 64 x 128 tiled weights
    # GEMV: M outside [1, 16] is unsupported, bad dtype unsupported, misaligned
    assert lib.q4_gemv(fake, 1, 0, 64, 128, fake, TILED, wb, fake, 0, None, 0, None) == 2
    assert lib.q4_gemv(fake, 1, 17, 64, 128, fake, TILED, wb, fake, 0, None, 0, None) == 2
    assert lib.q4_gemv(fake, 7, 1, 64, 128, fake, TILED, wb, fake, 0, None, 0, None) == 2
    assert lib.q4_gemv(fake + 2, 1, 1, 64, 128, fake, TILED, wb, fake, 0, None, 0, None) == 3
    assert lib.q4_gemv(fake, 1, 1, 64, 129, fake, TILED, wb, fake, 0, None, 0, None) == 1
    # the CUDA-core path takes M = 1 and the tiled layout only
    assert lib.q4_gemv_path(fake, 1, 2, 64, 128, fake, TILED, wb, fake, 0, None, 0, 1, None) == 2
    assert lib.q4_gemv_path(fake, 1, 1, 64, 128, fake, COMPACT, 4 * 1072, fake, 0, None, 0, 1,
                            None) == 2


@pytest.mark.parametrize("fn", ["q4_gemv", "q4_gemm", "q4_gemv_timeout_selftest",
                                "q4_gemm_timeout_selftest"])
def test_weight_layout_is_checked_before_any_launch(lib, fn):
    """A weight buffer must match its declared layout and shape byte for
    byte: compact tiles handed over as tiled ones (or the reverse), a buffer
    for another shape, or an unknown layout are refused with INVALID_ARG
    before anything touches the GPU."""
    _product_argtypes(lib)
    f = getattr(lib, fn)
    fake = 4096
    N, K = 64, 256
    tiled, compact = 4 * 2 * 1104, 4 * 2 * 1072
    for layout, nb in ((TILED, compact), (COMPACT, tiled), (TILED, tiled + 16), (TILED, 0),
                       (0, tiled), (3, compact), (TILED, 4 * 1 * 1104)):
        assert f(fake, 1, 1, N, K, fake, layout, nb, fake, 1, None, 0, None) == 1, (layout, nb)
    lib.q4_gemv_noalloc.restype = ctypes.c_int
    assert lib.q4_gemv_noalloc(fake, 1, 1, N, K, fake, TILED, compact, fake, 1, None) == 1


def test_gemm_host_side_errors(lib):
    _product_argtypes(lib)
    fake = 4096
    wb = 4 * 1104
    # f32 activations are not taken by the tensor-core GEMM
    assert lib.q4_gemm(fake, 0, 4, 64, 128, fake, TILED, wb, fake, 1, None, 0, None) == 2
    assert lib.q4_gemm(fake, 1, 0, 64, 128, fake, TILED, wb, fake, 1, None, 0, None) == 1
    assert lib.q4_gemm(fake + 8, 1, 4, 64, 128, fake, TILED, wb, fake, 1, None, 0, None) == 3
    assert lib.q4_gemm(fake, 1, 4, 64, 100, fake, TILED, wb, fake, 1, None, 0, None) == 1
