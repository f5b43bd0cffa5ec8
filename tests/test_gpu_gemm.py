"""Large-M W4A16 GEMM (tcgen05) through the C ABI against the oracle's plain
dequantize-then-dot, element by element, under the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_bf16_bits, dev_f32, oracle_product, x_for

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(256, 128, 512), (300, 144, 1024), (513, 384, 1024),
                                   (64, 256, 2048), (1000, 1024, 4096)])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_gemm_parity(M, N, K, xdt):
    import weight_only_int4_group_gb300 as q4
    W = synth.normal_rows(M + N, K, 0, N, 0.02)
    x, xf = x_for(xdt, M, K, seed=M * 7 + K)
    _, y_ref, absdot = oracle_product(W, xf)
    qw = q4.QWeight.from_float(dev_f32(W))
    for ydt in (torch.bfloat16, torch.float16):
        y = q4.gemm(x, qw, out_dtype=ydt)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        compare(y, y_ref, absdot, where=f"gemm {M}x{N}x{K} y={ydt}")


@pytest.mark.parametrize("M", [1, 9, 16, 17, 32, 48, 64, 100, 128, 129, 255])
def test_gemm_small_m(M):
    """q4_gemm accepts any M >= 1; the token tile (16, 32, 64, 128 or 256
    rows) is the smallest that covers M, with a ragged last tile."""
    import weight_only_int4_group_gb300 as q4
    N, K = 384, 2048
    W = synth.normal_rows(M + 11, K, 0, N, 0.02)
    xdt = torch.float16 if M in (9, 100) else torch.bfloat16
    x, xf = x_for(xdt, M, K, seed=M + 3)
    _, y_ref, absdot = oracle_product(W, xf)
    y = q4.gemm(x, q4.QWeight.from_float(dev_f32(W)), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    compare(y, y_ref, absdot, where=f"gemm M={M}")


def test_gemm_outputs_untouched_beyond_bounds():
    """Ragged M and N: rows and columns past the matrix are not written."""
    import weight_only_int4_group_gb300 as q4
    M, N, K = 130, 160, 256
    W = synth.normal_rows(3, K, 0, N, 0.02)
    x, _ = x_for(torch.bfloat16, M, K, seed=5)
    qw = q4.QWeight.from_float(dev_f32(W))
    big = torch.full((M + 8, N), 9.0, dtype=torch.bfloat16, device="cuda")
    q4.gemm(x, qw, out=big[:M])
    torch.cuda.synchronize()
    assert bool((big[M:] == 9.0).all())


def test_gemm_rejects_bad_arguments():
    import weight_only_int4_group_gb300 as q4
    qw = q4.QWeight(torch.zeros(q4.weight_bytes(32, 128), dtype=torch.uint8, device="cuda"), 32, 128)
    x = torch.zeros((4, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.gemm(x, qw)
    assert ei.value.status == q4.ERR_UNSUPPORTED


def test_gemm_prefill_shape_sampled():
    """The prefill workload, 4096 x 8192 activations against 28672 x 8192
    weights (device-generated), sampled rows and columns against the oracle."""
    import weight_only_int4_group_gb300 as q4
    M, N, K = 4096, 28672, 8192
    seed = 301
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    synth.dev_normal_f32(w.data_ptr(), N * K, seed, 0, 0.02)
    qw = q4.QWeight.from_float(w)
    del w
    xb = torch.empty(M * K, dtype=torch.int16, device="cuda")
    synth.dev_normal_bf16(xb.data_ptr(), M * K, seed + 1, 0, 1.0)
    x = xb.view(torch.bfloat16).view(M, K)
    y = q4.gemm(x, qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 12)]))
    ms = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 12)]))
    xbits = xb.view(M, K)[torch.from_numpy(ms).cuda()].cpu().numpy().view(np.uint16)
    xf = synth.bf16_bits_to_f32(xbits)
    o = oracle.load()
    for r in rows:
        Wr = synth.normal_rows(seed, K, int(r), int(r) + 1, 0.02)
        p, s, z = o.quantize(Wr)
        yr, ar = o.dot_naive(xf, p, s, z, 1, K)
        compare(y[torch.from_numpy(ms).cuda(), int(r):int(r) + 1], yr, ar, where=f"row {r}")
