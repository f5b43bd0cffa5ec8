"""Canary tests: no entry point writes outside the buffers it is given.

Every output buffer (and every workspace) is placed inside a larger
allocation whose bytes on either side are filled with a guard pattern; after
the call the guards must be intact, the inputs unchanged, q4_check must
report OK and a workspace must be back to all zeros.  The shapes are ragged
(row counts that end inside a 16-row tile, token counts that end inside a
batch tile) and cover the split-K paths of both products, where partial sums
and arrival counters are written.

The same file, together with the parity suites, is run once more in a child
process against libq4_debug.so (built with -DQ4_DEBUG), in which every
global store of every kernel is checked against its buffer's extent: an
out-of-range store is recorded and skipped, and q4_check returns
Q4_ERR_BOUNDS.  Those checks see stores that land inside other live memory,
which guard bytes cannot."""
from __future__ import annotations

import os
import re
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import dev_f32, x_for

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DEBUG_LIB = os.path.join(ROOT, "weight_only_int4_group_gb300", "libq4_debug.so")
UNDER_DEBUG = os.path.abspath(os.environ.get("Q4_LIBRARY", "")) == DEBUG_LIB
PAD = 4096  # guard bytes on each side (keeps every view 16-byte aligned)
GUARD = 0xA5


def q4():
    import weight_only_int4_group_gb300 as m
    return m


def stream() -> int:
    return torch.cuda.current_stream().cuda_stream


class Guarded:
    """`nbytes` of device memory with PAD guard bytes on either side."""

    def __init__(self, nbytes: int, fill: int = GUARD):
        self.n = nbytes
        self.buf = torch.full((PAD + nbytes + PAD,), GUARD, dtype=torch.uint8, device="cuda")
        self.buf[PAD:PAD + nbytes] = fill

    def view(self, dtype=torch.uint8, shape=None) -> torch.Tensor:
        v = self.buf[PAD:PAD + self.n].view(dtype)
        return v.view(shape) if shape is not None else v

    def ptr(self) -> int:
        return self.buf.data_ptr() + PAD

    def assert_guards(self, what: str):
        lo = self.buf[:PAD].cpu().numpy()
        hi = self.buf[PAD + self.n:].cpu().numpy()
        bad_lo = np.flatnonzero(lo != GUARD)
        bad_hi = np.flatnonzero(hi != GUARD)
        assert bad_lo.size == 0, f"{what}: {bad_lo.size} bytes written below the buffer " \
                                 f"(nearest at offset {int(bad_lo[-1]) - PAD})"
        assert bad_hi.size == 0, f"{what}: {bad_hi.size} bytes written past the buffer " \
                                 f"(first at offset +{int(bad_hi[0])})"


def ok(rc: int, what: str):
    assert rc == q4().OK, f"{what}: status {rc}"


def checked(what: str):
    rc = q4().check()
    assert rc == q4().OK, f"{what}: q4_check returned {rc}"


def weights(N: int, K: int, seed: int, compact: bool = False):
    W = synth.normal_rows(seed, K, 0, N, 0.02)
    return q4().QWeight.from_float(dev_f32(W), compact=compact)


# ----------------------------------------------------------------- packing
@pytest.mark.parametrize("N,K", [(1000, 1024), (37, 384), (1, 128)])
@pytest.mark.parametrize("sym", [False, True])
def test_quantize_stays_inside(N, K, sym):
    m = q4()
    W = dev_f32(synth.normal_rows(3, K, 0, N, 0.02))
    W0 = W.clone()
    G = K // 128
    packed, scale, zero = Guarded(N * K // 2), Guarded(N * G * 4), Guarded(N * G)
    fn = m.lib().q4_quantize_sym if sym else m.lib().q4_quantize
    ok(fn(W.data_ptr(), N, K, packed.ptr(), scale.ptr(), zero.ptr(), stream()), "quantize")
    checked("quantize")
    for b, n in ((packed, "packed"), (scale, "scale"), (zero, "zero")):
        b.assert_guards(f"quantize {n} {N}x{K}")
    assert torch.equal(W, W0)
    ref = m.quantize_sym(W) if sym else m.quantize(W)
    assert torch.equal(packed.view(torch.uint8, (N, K // 2)), ref[0])
    assert torch.equal(scale.view(torch.float32, (N, G)), ref[1])
    assert torch.equal(zero.view(torch.uint8, (N, G)), ref[2])


@pytest.mark.parametrize("N,K", [(1000, 1024), (37, 384), (1, 128), (16, 256)])
@pytest.mark.parametrize("compact", [False, True])
def test_repack_unpack_stay_inside(N, K, compact):
    m = q4()
    lib = m.lib()
    W = dev_f32(synth.normal_rows(5, K, 0, N, 0.02))
    packed, scale, zero = m.quantize(W)
    ins = [t.clone() for t in (packed, scale, zero)]
    layout = m.LAYOUT_COMPACT if compact else m.LAYOUT_TILED
    nb = m.weight_bytes(N, K, layout)
    qw = Guarded(nb, fill=0)
    fn = lib.q4_repack_compact if compact else lib.q4_repack
    ok(fn(packed.data_ptr(), scale.data_ptr(), zero.data_ptr(), N, K, qw.ptr(), stream()),
       "repack")
    checked("repack")
    qw.assert_guards(f"repack {N}x{K} compact={compact}")
    for a, b in zip(ins, (packed, scale, zero)):
        assert torch.equal(a, b)
    qw_copy = qw.view().clone()

    G = K // 128
    p2, s2, z2 = Guarded(N * K // 2), Guarded(N * G * (2 if compact else 4)), Guarded(N * G)
    fn = lib.q4_unpack_compact if compact else lib.q4_unpack
    ok(fn(qw.ptr(), N, K, p2.ptr(), s2.ptr(), z2.ptr(), stream()), "unpack")
    checked("unpack")
    for b, n in ((p2, "packed"), (s2, "scale"), (z2, "zero")):
        b.assert_guards(f"unpack {n} {N}x{K} compact={compact}")
    assert torch.equal(qw.view(), qw_copy)
    assert torch.equal(p2.view(torch.uint8, (N, K // 2)), packed)
    assert torch.equal(z2.view(torch.uint8, (N, G)), zero)
    if not compact:
        assert torch.equal(s2.view(torch.float32, (N, G)), scale)


@pytest.mark.parametrize("M,K", [(1, 128), (3, 4096), (17, 1152)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_xsum_stays_inside(M, K, dtype):
    m = q4()
    x, _ = x_for(dtype, M, K, seed=9)
    x0 = x.clone()
    out = Guarded(M * (K // 128) * 4)
    ok(m.lib().q4_xsum(x.data_ptr(), m._DTYPE[dtype], M, K, out.ptr(), stream()), "xsum")
    checked("xsum")
    out.assert_guards(f"xsum M={M} K={K}")
    assert torch.equal(x, x0)
    assert torch.equal(out.view(torch.float32, (M, K // 128)), m.xsum(x))


# ----------------------------------------------------------------- products
def run_product(fn_name, x, qw, M, out_dtype):
    """One call with guarded y and workspace; returns y (a view)."""
    m = q4()
    lib = m.lib()
    esz = torch.tensor([], dtype=out_dtype).element_size()
    y = Guarded(M * qw.N * esz, fill=0x7F)
    need = (m.gemv_workspace_bytes if fn_name == "gemv" else m.gemm_workspace_bytes)(M, qw.N, qw.K)
    ws = Guarded(need, fill=0) if need else None
    x0, qw0 = x.clone(), qw.data.clone()
    fn = lib.q4_gemv if fn_name == "gemv" else lib.q4_gemm
    ok(fn(x.data_ptr(), m._DTYPE[x.dtype], M, qw.N, qw.K, qw.data.data_ptr(), qw.layout, qw.nbytes,
          y.ptr(), m._DTYPE[out_dtype], ws.ptr() if ws else 0, need, stream()), fn_name)
    checked(fn_name)
    what = f"{fn_name} M={M} N={qw.N} K={qw.K}"
    y.assert_guards(what + " y")
    if ws is not None:
        ws.assert_guards(what + " workspace")
        assert int(torch.count_nonzero(ws.view())) == 0, what + ": workspace not left zero"
    assert torch.equal(x, x0) and torch.equal(qw.data, qw0), what + ": an input changed"
    return y.view(out_dtype, (M, qw.N))


@pytest.mark.parametrize("N,K", [(1000, 8192), (3000, 4096), (8, 28672)])
@pytest.mark.parametrize("M", [1, 2, 5, 9, 16])
def test_gemv_stays_inside(N, K, M):
    m = q4()
    compact = M in (2, 9)
    qw = weights(N, K, 11 + M, compact=compact)
    for xdt, ydt in ((torch.bfloat16, torch.float32), (torch.float16, torch.bfloat16),
                     (torch.float32, torch.float16)):
        x, _ = x_for(xdt, M, K, seed=M)
        y = run_product("gemv", x, qw, M, ydt)
        ref = m.gemv(x, qw, out_dtype=ydt)
        assert torch.equal(y, ref), f"gemv M={M} {xdt}->{ydt}: differs from a plain call"


def test_gemv_noalloc_stays_inside():
    m = q4()
    lib = m.lib()
    M, N, K = 3, 1000, 8192
    qw = weights(N, K, 21)
    x, _ = x_for(torch.bfloat16, M, K, seed=4)
    y = Guarded(M * N * 4, fill=0x7F)
    ok(lib.q4_gemv_noalloc(x.data_ptr(), m.BF16, M, N, K, qw.data.data_ptr(), qw.layout, qw.nbytes,
                           y.ptr(), m.F32, stream()), "gemv_noalloc")
    checked("gemv_noalloc")
    y.assert_guards("gemv_noalloc y")
    assert torch.equal(y.view(torch.float32, (M, N)), m.gemv(x, qw, out_dtype=torch.float32))


@pytest.mark.parametrize("M,N,K", [(1, 1000, 8192), (37, 1000, 4096), (130, 200, 1024),
                                   (300, 1000, 2048), (64, 8, 28672)])
def test_gemm_stays_inside(M, N, K):
    m = q4()
    for compact, xdt, ydt in ((False, torch.bfloat16, torch.float32),
                              (True, torch.float16, torch.bfloat16)):
        qw = weights(N, K, 31 + M, compact=compact)
        x, _ = x_for(xdt, M, K, seed=M + 1)
        y = run_product("gemm", x, qw, M, ydt)
        ref = m.gemm(x, qw, out_dtype=ydt)
        assert torch.equal(y, ref), f"gemm M={M} N={N} K={K}: differs from a plain call"


# ----------------------------------------------------------------- debug build
def test_debug_bounds_selftest():
    """The release library refuses the self-test; the debug library records a
    store outside the declared extent and skips it."""
    m = q4()
    buf = torch.zeros(32, dtype=torch.uint8, device="cuda")
    rc = m.lib().q4_debug_bounds_selftest(buf.data_ptr(), stream())
    if not UNDER_DEBUG:
        assert rc == m.ERR_UNSUPPORTED
        checked("selftest (release)")
        assert int(torch.count_nonzero(buf)) == 0
        return
    assert rc == m.OK
    assert m.check() == m.ERR_BOUNDS
    assert buf.cpu().tolist() == list(range(1, 17)) + [0] * 16
    checked("after the self-test")  # the error word was cleared


PARITY_UNDER_DEBUG = ["tests/test_gpu_canaries.py", "tests/test_gpu_quantize.py",
                      "tests/test_gpu_quantize_sym.py", "tests/test_gpu_compact.py",
                      "tests/test_gpu_gemv.py", "tests/test_gpu_gemm.py",
                      "tests/test_gpu_fullsize.py", "tests/test_gpu_random_shapes.py",
                      "tests/test_zz_no_alloc.py"]


@pytest.mark.skipif(UNDER_DEBUG, reason="already running against the debug library")
def test_parity_suites_under_debug_build():
    """Runs the canary and parity suites again in a child process against
    libq4_debug.so.  Every GPU test there ends with a q4_check that must not
    report Q4_ERR_BOUNDS (see conftest), and the self-test above proves the
    debug library was the one loaded."""
    assert os.path.exists(DEBUG_LIB), "libq4_debug.so is missing: run __graft_entry__.build()"
    env = dict(os.environ, Q4_LIBRARY=DEBUG_LIB)
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           *PARITY_UNDER_DEBUG]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-4000:]
    assert r.returncode == 0, tail
    passed = re.search(r"(\d+) passed", r.stdout)
    assert passed and "failed" not in r.stdout, tail
    # every collected test ran (the suites hold about four hundred)
    assert int(passed.group(1)) >= 300, tail
