"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: weights drawn on the device by the counter-based generator,
quantized and packed by the library, multiplied by the GEMV; sampled rows are
regenerated on the host and checked against the oracle (codes bit-exact,
outputs under the tolerance)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_bf16_bits

pytestmark = pytest.mark.gpu

SIGMA = 0.02


def _device_weights(N, K, seed, cols=None):
    w = torch.empty((N, K), dtype=torch.float32, device="cuda")
    mask = None
    if cols is not None and len(cols):
        m = np.zeros(K, np.uint8)
        m[cols] = 1
        mask = torch.from_numpy(m).cuda()
    synth.dev_normal_f32(w.data_ptr(), N * K, seed, 0, SIGMA,
                         mask.data_ptr() if mask is not None else 0, K, 20.0)
    return w


def _check_sampled(N, K, M, seed, cols=None, nsample=24, product="gemv"):
    import weight_only_int4_group_gb300 as q4
    w = _device_weights(N, K, seed, cols)
    packed, scale, zero = q4.quantize(w)
    del w
    qw = q4.QWeight(q4.repack(packed, scale, zero, N, K), N, K)
    xbits = synth.normal_bf16(seed + 1, 0, M * K).reshape(M, K)
    x = dev_bf16_bits(xbits)
    y = (q4.gemv if product == "gemv" else q4.gemm)(x, qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK

    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, nsample)]))
    o = oracle.load()
    xf = synth.bf16_bits_to_f32(xbits)
    c = np.zeros(0, np.int32) if cols is None else cols
    for r in rows:
        Wr = synth.normal_rows(seed, K, int(r), int(r) + 1, SIGMA, c, 20.0)
        pr, sr, zr = o.quantize(Wr)
        assert np.array_equal(packed[r].cpu().numpy(), pr[0]), f"codes of row {r}"
        assert np.array_equal(scale[r].cpu().numpy().view(np.uint32), sr[0].view(np.uint32))
        assert np.array_equal(zero[r].cpu().numpy(), zr[0])
        yr, ar = o.dot_naive(xf, pr, sr, zr, 1, K)
        compare(y[:, r:r + 1], yr, ar, where=f"{N}x{K} M={M} row {r}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_70b_mlp_up(M):
    _check_sampled(28672, 8192, M, seed=101)


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_70b_mlp_down(M):
    _check_sampled(8192, 28672, M, seed=102)


@pytest.mark.parametrize("N,K", [(28672, 8192), (8192, 28672)])
def test_70b_mlp_m32_gemm(N, K):
    """The batch sweep's M = 32 point, which goes through q4_gemm (few
    tiles: the groups are split over the CTAs)."""
    _check_sampled(N, K, 32, seed=103 + K, product="gemm")


def test_70b_fused_gate_up():
    _check_sampled(57344, 8192, 1, seed=103, nsample=16)


@pytest.mark.parametrize("N,K", [(12288, 4096), (4096, 4096), (11008, 4096), (4096, 11008)])
def test_7b_layer_with_outliers(N, K):
    cols = synth.outlier_columns(200 + K, K)
    _check_sampled(N, K, 1, seed=N + K, cols=cols)


def test_7b_gate_up_rows_concatenated():
    """Gate and up quantized separately and their tiled buffers concatenated
    along the rows (11008 is a whole number of 16-row tiles): one 22016 x
    4096 GEMV, as the 7B layer benchmark runs it; sampled rows of both halves
    against the oracle, each half with its own outlier columns."""
    import weight_only_int4_group_gb300 as q4
    K, Nh = 4096, 11008
    parts, meta = [], []
    for h, seed in enumerate((301, 302)):
        cols = synth.outlier_columns(210 + h, K)
        w = _device_weights(Nh, K, seed, cols)
        parts.append(q4.QWeight.from_float(w))
        meta.append((seed, cols))
        del w
    fused = q4.QWeight(torch.cat([parts[0].data, parts[1].data]), 2 * Nh, K)
    assert fused.nbytes == q4.weight_bytes(2 * Nh, K)
    xbits = synth.normal_bf16(303, 0, K).reshape(1, K)
    y = q4.gemv(dev_bf16_bits(xbits), fused, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    o = oracle.load()
    xf = synth.bf16_bits_to_f32(xbits)
    rng = np.random.default_rng(304)
    for h, (seed, cols) in enumerate(meta):
        for r in np.unique(np.concatenate([[0, Nh - 1], rng.integers(0, Nh, 12)])):
            Wr = synth.normal_rows(seed, K, int(r), int(r) + 1, SIGMA, cols, 20.0)
            pr, sr, zr = o.quantize(Wr)
            yr, ar = o.dot_naive(xf, pr, sr, zr, 1, K)
            col = h * Nh + int(r)
            compare(y[:, col:col + 1], yr, ar, where=f"half {h} row {r}")


def test_device_generator_matches_host():
    n = 1 << 16
    t = torch.empty(n, dtype=torch.float32, device="cuda")
    synth.dev_normal_f32(t.data_ptr(), n, 77, 12345, 0.02)
    host = synth.normal(77, 12345, n, 0.02)
    assert np.array_equal(t.cpu().numpy().view(np.uint32), host.view(np.uint32))
    b = torch.empty(n, dtype=torch.int16, device="cuda")
    synth.dev_normal_bf16(b.data_ptr(), n, 78, 5)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), synth.normal_bf16(78, 5, n))
    synth.dev_uniform_f32(t.data_ptr(), n, 79, 0, 0.5)
    assert np.array_equal(t.cpu().numpy().view(np.uint32), synth.uniform(79, 0, n, 0.5).view(np.uint32))
