"""q4_gemv_noalloc: the GEMV entry point for callers that cannot allocate
device memory (a plugin whose host framework owns every device buffer and
hands over only inputs and outputs, a decode loop that must never call an
allocator): it takes its workspace from a static scratch array inside the
library instead of from the caller.

Called through the C ABI and checked against q4_gemv (caller-provided
workspace) and against the oracle, on two calls in a row, so the second call
runs on scratch left behind by the first; and on a sequence of different
output sizes sharing the one array.  Kept in a file of its own, named to be
collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import RTOL, ATOL, compare, dev_bf16_bits, dev_f32

pytestmark = pytest.mark.gpu

P, I, Z, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int


def _lib():
    import weight_only_int4_group_gb300 as q4
    lib = q4.lib()
    lib.q4_gemv_noalloc.argtypes = [P, S, I, I, I, P, S, Z, P, S, P]
    lib.q4_gemv_noalloc.restype = S
    return lib


def _problem(N, K, M, seed):
    import weight_only_int4_group_gb300 as q4
    W = synth.normal_rows(seed, K, 0, N, 0.02)
    qw = q4.QWeight.from_float(dev_f32(W))
    bits = synth.normal_bf16(seed + 1, 0, M * K).reshape(M, K)
    o = oracle.load()
    p, s, z = o.quantize(W)
    y_ref, absdot = o.dot_naive(synth.bf16_bits_to_f32(bits), p, s, z, N, K, threads=16)
    return qw, dev_bf16_bits(bits), y_ref, absdot


def _noalloc(lib, x, qw, M):
    import weight_only_int4_group_gb300 as q4
    y = torch.full((M, qw.N), float("nan"), device="cuda")
    rc = lib.q4_gemv_noalloc(x.data_ptr(), q4.BF16, M, qw.N, qw.K, qw.data.data_ptr(), qw.layout,
                             qw.nbytes, y.data_ptr(), q4.F32,
                             torch.cuda.current_stream().cuda_stream)
    assert rc == q4.OK, rc
    return y


@pytest.mark.parametrize("N,K,M", [(8192, 28672, 1), (3000, 4096, 4), (1000, 8192, 16)])
def test_noalloc_matches_gemv_twice(N, K, M):
    import weight_only_int4_group_gb300 as q4
    lib = _lib()
    qw, x, y_ref, absdot = _problem(N, K, M, 31)
    assert q4.gemv_workspace_bytes(M, N, K) <= 16 << 20  # within the static scratch
    tol = RTOL * absdot + ATOL
    for _ in range(2):
        ref = q4.gemv(x, qw, out_dtype=torch.float32)  # caller-provided workspace
        y = _noalloc(lib, x, qw, M)
        assert q4.check() == q4.OK
        err = np.abs(y.cpu().numpy().astype(np.float64) - ref.cpu().numpy().astype(np.float64))
        assert (err <= tol).all(), float((err / tol).max())
        compare(y, y_ref, absdot, where=f"noalloc {N}x{K} M={M}")


def test_noalloc_scratch_used_across_output_sizes():
    """Calls with N = 8192, then 3000, then 8192 again share the one static
    array (each needs a split over K, so the scratch is really used); every
    result matches q4_gemv and the oracle."""
    import weight_only_int4_group_gb300 as q4
    lib = _lib()
    probs = {N: _problem(N, K, 1, 40 + N % 7) for N, K in ((8192, 28672), (3000, 4096))}
    for N, (qw, _, _, _) in probs.items():
        assert q4.gemv_workspace_bytes(1, N, qw.K) > 0, N
    for N in (8192, 3000, 8192):
        qw, x, y_ref, absdot = probs[N]
        y = _noalloc(lib, x, qw, 1)
        ref = q4.gemv(x, qw, out_dtype=torch.float32)
        assert q4.check() == q4.OK
        assert torch.equal(y, ref), N
        compare(y, y_ref, absdot, where=f"noalloc sequence N={N}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import weight_only_int4_group_gb300 as q4
    lib = _lib()
    M, N, K = 16, 1 << 22, 8192  # would need far more than the static scratch
    assert q4.gemv_workspace_bytes(M, N, K) > 16 << 20
    fake = 4096  # never dereferenced: rejected before any launch
    rc = lib.q4_gemv_noalloc(fake, q4.BF16, M, N, K, fake, q4.LAYOUT_TILED,
                             q4.weight_bytes(N, K), fake, q4.F32,
                             torch.cuda.current_stream().cuda_stream)
    assert rc == q4.ERR_UNSUPPORTED
    assert q4.check() == q4.OK
