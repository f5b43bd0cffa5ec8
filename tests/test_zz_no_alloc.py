"""q4_gemv_noalloc: the GEMV entry point for callers that cannot allocate
device memory (it takes its workspace from a static scratch array in the
library instead of from the caller).  Called through the C ABI and checked
against q4_gemv (caller-provided workspace) on two calls in a row, so the
second call runs on scratch left behind by the first.  Kept in a file of its
own, named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import RTOL, ATOL, dev_bf16_bits, dev_f32

pytestmark = pytest.mark.gpu

P, I, Z, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int


def _lib():
    import weight_only_int4_group_gb300 as q4
    lib = q4.lib()
    lib.q4_gemv_noalloc.argtypes = [P, S, I, I, I, P, P, S, P]
    lib.q4_gemv_noalloc.restype = S
    return lib


@pytest.mark.parametrize("N,K,M", [(8192, 28672, 1), (3000, 4096, 4), (1000, 8192, 16)])
def test_noalloc_matches_gemv_twice(N, K, M):
    import weight_only_int4_group_gb300 as q4
    lib = _lib()
    W = synth.normal_rows(31, K, 0, N, 0.02)
    qw = q4.QWeight.from_float(dev_f32(W))
    bits = synth.normal_bf16(32, 0, M * K).reshape(M, K)
    x = dev_bf16_bits(bits)
    p, s, z = oracle.load().quantize(W)
    _, absdot = oracle.load().dot_naive(synth.bf16_bits_to_f32(bits), p, s, z, N, K, threads=8)
    tol = RTOL * absdot + ATOL
    assert q4.gemv_workspace_bytes(M, N, K) <= 16 << 20
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        ref = q4.gemv(x, qw, out_dtype=torch.float32)  # caller-provided workspace
        y = torch.full((M, N), float("nan"), device="cuda")
        rc = lib.q4_gemv_noalloc(x.data_ptr(), q4.BF16, M, N, K, qw.data.data_ptr(),
                                 y.data_ptr(), q4.F32, stream)
        assert rc == q4.OK
        assert q4.check() == q4.OK
        err = np.abs(y.cpu().numpy().astype(np.float64) - ref.cpu().numpy().astype(np.float64))
        assert (err <= tol).all(), float((err / tol).max())


def test_noalloc_rejects_problems_beyond_its_scratch():
    import weight_only_int4_group_gb300 as q4
    lib = _lib()
    M, N, K = 16, 1 << 22, 8192  # would need far more than the static scratch
    assert q4.gemv_workspace_bytes(M, N, K) > 16 << 20
    fake = 4096  # never dereferenced: rejected before any launch
    rc = lib.q4_gemv_noalloc(fake, q4.BF16, M, N, K, fake, fake, q4.F32,
                             torch.cuda.current_stream().cuda_stream)
    assert rc == q4.ERR_UNSUPPORTED
    assert q4.check() == q4.OK
