"""GPU symmetric quantizer (q4_quantize_sym) against the oracle: codes, scales
and zeros bit-exact, including ties, near-ties and underflowing scales; the
page's own synthetic matrix and its printed error figures; GEMV and GEMM on
symmetric weights under the product tolerance; a full-size sampled check."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_bf16_bits, dev_f32, x_for
from test_gpu_quantize import _edge_matrix

pytestmark = pytest.mark.gpu


def _sym_edge_matrix(N, K, seed):
    W = _edge_matrix(N, K, seed)
    if N >= 16:
        rng = np.random.default_rng(seed + 1)
        W[12] = rng.integers(-7, 8, K).astype(np.float32)   # max|w| = 7: scale exactly 1
        W[12, ::128] = 7.0
        W[12, 1::5] = 2.5                                     # exact ties of w / scale
        W[12, 2::5] = -3.5
        W[12, 3::11] = 6.5
        W[13] = np.float32(np.ldexp(1.0, -149))               # max|w|/7 underflows: scale 1
        W[14] = np.float32(np.ldexp(6.0, -149))               # subnormal scale
        W[14, 5::9] = np.float32(np.ldexp(-3.0, -149))
        W[15] = -W[15]                                        # a sign flip of ordinary data
    return W


def _check_exact(W):
    import weight_only_int4_group_gb300 as q4
    p, s, z = q4.quantize_sym(dev_f32(W))
    torch.cuda.synchronize()
    po, so, zo = oracle.load().quantize(W, symmetric=True)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zo)
    assert np.array_equal(p.cpu().numpy(), po)
    return p, s, z


@pytest.mark.parametrize("N,K", [(1, 128), (2, 256), (16, 128), (200, 1024), (33, 4096),
                                 (16, 11008)])
def test_quantize_sym_bit_exact(N, K):
    _check_exact(_sym_edge_matrix(N, K, seed=N * 13 + K))


def test_quantize_sym_near_tie_quotients():
    """Weights whose quotient w / scale lies within a few ulps of n + 1/2:
    the codes must follow the IEEE f32 quotient with ties to even."""
    rng = np.random.default_rng(29)
    N, K = 64, 1024
    W = np.empty((N, K), dtype=np.float32)
    for r in range(N):
        for g in range(K // 128):
            a = np.float32(rng.uniform(0.01, 1.0))
            s = np.float32(a / np.float32(7.0))
            n = rng.integers(-7, 7, 127).astype(np.float32)
            w = np.float32((n + np.float32(0.5)) * s)
            steps = rng.integers(-3, 4, 127)
            for i, k in enumerate(steps):
                for _ in range(abs(int(k))):
                    w[i] = np.nextafter(w[i], np.float32(np.inf if k > 0 else -np.inf))
            w = np.clip(w, -a, a)
            W[r, g * 128:(g + 1) * 128] = np.concatenate([[a if r % 2 else -a], w])
    _check_exact(W)


def test_quantize_sym_page_matrix():
    """The page's 256 x 1024 synthetic matrix: bit-exact, and the group-128
    error the page prints (18.2 dB, 12.24 %) recomputed from the GPU's
    codes and scales."""
    w = synth.row_scaled_outliers()
    p, s, z = _check_exact(w.astype(np.float32))
    wh = oracle.load().dequant(p.cpu().numpy(), s.cpu().numpy(), z.cpu().numpy(), 256, 1024)
    sig, err = float((w * w).sum()), float(((w - wh) ** 2).sum())
    assert f"{10 * np.log10(sig / err):.1f}" == "18.2"
    assert f"{100 * np.sqrt(err / sig):.2f}" == "12.24"


@pytest.mark.parametrize("M", [1, 5, 16])
def test_gemv_on_symmetric_weights(M):
    import weight_only_int4_group_gb300 as q4
    N, K = 1000, 2048
    W = np.random.default_rng(M).normal(0, 0.02, (N, K)).astype(np.float32)
    qw = q4.QWeight.from_float(dev_f32(W), symmetric=True)
    x, xf = x_for(torch.bfloat16, M, K, seed=40 + M)
    y = q4.gemv(x, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    o = oracle.load()
    p, s_, z = o.quantize(W, symmetric=True)
    yr, ar = o.dot_naive(xf, p, s_, z, N, K, threads=8)
    compare(y, yr, ar, where=f"sym gemv M={M}")


def test_gemm_on_symmetric_weights():
    import weight_only_int4_group_gb300 as q4
    M, N, K = 300, 384, 1024
    W = np.random.default_rng(3).normal(0, 0.02, (N, K)).astype(np.float32)
    qw = q4.QWeight.from_float(dev_f32(W), symmetric=True)
    x, xf = x_for(torch.bfloat16, M, K, seed=44)
    y = q4.gemm(x, qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    o = oracle.load()
    p, s_, z = o.quantize(W, symmetric=True)
    yr, ar = o.dot_naive(xf, p, s_, z, N, K, threads=8)
    compare(y, yr, ar, where="sym gemm")


def test_quantize_sym_fullsize_sampled():
    """28672 x 8192 drawn on the device (the 70B up-projection shape), in the
    launch configuration the benchmark times; sampled rows bit-exact."""
    import weight_only_int4_group_gb300 as q4
    from test_gpu_fullsize import SIGMA, _device_weights
    N, K, seed = 28672, 8192, 131
    w = _device_weights(N, K, seed)
    p, s, z = q4.quantize_sym(w)
    del w
    qw = q4.QWeight(q4.repack(p, s, z, N, K), N, K)
    xbits = synth.normal_bf16(seed + 1, 0, K).reshape(1, K)
    y = q4.gemv(dev_bf16_bits(xbits), qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    o = oracle.load()
    xf = synth.bf16_bits_to_f32(xbits)
    rng = np.random.default_rng(seed)
    for r in np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 16)])):
        Wr = synth.normal_rows(seed, K, int(r), int(r) + 1, SIGMA)
        pr, sr, zr = o.quantize(Wr, symmetric=True)
        assert np.array_equal(p[r].cpu().numpy(), pr[0]), f"codes of row {r}"
        assert np.array_equal(s[r].cpu().numpy().view(np.uint32), sr[0].view(np.uint32))
        assert np.array_equal(z[r].cpu().numpy(), zr[0])
        yr, ar = o.dot_naive(xf, pr, sr, zr, 1, K)
        compare(y[:, r:r + 1], yr, ar, where=f"sym {N}x{K} row {r}")
