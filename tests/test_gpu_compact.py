"""Compact tiles (binary16 scales, 4-bit zeros) against the oracle: the
repack's codes, scale bits and zeros bit-exact (unpacked), the GEMV under the
product tolerance with the oracle's expanded metadata, and a full-size
sampled check."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_bf16_bits, dev_f32, x_for

pytestmark = pytest.mark.gpu


def _oracle_compact(W):
    """Oracle codes, binary16 scale bits, zeros and the expanded scales."""
    o = oracle.load()
    p, s, z = o.quantize(W)
    s16, z4 = o.compact_meta(s, z)
    se, ze = o.expand_meta(s16, z4, s.shape[1])
    assert np.array_equal(ze, z)
    return p, s16, z, se


@pytest.mark.parametrize("N,K", [(1, 128), (15, 256), (16, 128), (17, 384), (200, 1024),
                                 (33, 4096)])
def test_repack_compact_bit_exact(N, K):
    import weight_only_int4_group_gb300 as q4
    rng = np.random.default_rng(N * 5 + K)
    W = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    if N > 3:
        W[1] *= np.float32(50.0)      # large scales
        W[2] *= np.float32(0.05)      # small ones (still normal binary16)
    packed, scale, zero = q4.quantize(dev_f32(W))
    qw = q4.repack_compact(packed, scale, zero, N, K)
    assert qw.numel() == q4.weight_bytes_compact(N, K) == ((N + 15) // 16) * (K // 128) * 1072
    p2, s16, z2 = q4.unpack_compact(qw, N, K)
    torch.cuda.synchronize()
    po, so16, zo, _ = _oracle_compact(W)
    assert np.array_equal(p2.cpu().numpy(), po)
    assert np.array_equal(s16.cpu().numpy().view(np.uint16), so16)
    assert np.array_equal(z2.cpu().numpy(), zo)
    if N % 16:  # rows past N in the last tile are zero, padding included
        # the last row tile's tiles, by the tile order include/q4.h states
        T, NG = (N + 15) // 16, K // 128
        b = (T - 1) // 8
        nb = min(8, T - 8 * b)
        tiles = qw.view(T * NG, 1072).cpu().numpy()
        t = np.stack([tiles[8 * NG * b + nb * 4 * (g // 4) + (T - 1 - 8 * b) * min(4, NG - 4 * (g // 4))
                            + g % 4] for g in range(NG)])
        sp = t[:, 1024:1056].view(np.uint16).reshape(NG, 8, 2)
        for r in range(N % 16, 16):
            assert (sp[:, r % 8, r // 8] == 0).all()
        assert (t[:, 1064:] == 0).all()


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float16, torch.float32],
                         ids=["bf16", "f16", "f32"])
def test_gemv_compact_parity(M, xdt):
    import weight_only_int4_group_gb300 as q4
    N, K = 1000, 2944  # ragged rows (not a multiple of 128), K not a multiple of 512
    W = synth.normal_rows(M + 70, K, 0, N, 0.02)
    x, xf = x_for(xdt, M, K, seed=M + 90)
    qw = q4.QWeight.from_float(dev_f32(W), compact=True)
    y = q4.gemv(x, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    p, _, z, se = _oracle_compact(W)
    yr, ar = oracle.load().dot_naive(xf, p, se, z, N, K, threads=8)
    compare(y, yr, ar, where=f"compact gemv M={M} x={xdt}")


def test_gemv_compact_many_steps_per_cta():
    """A launch long enough for the 3-stage M = 1 ring and split row blocks."""
    import weight_only_int4_group_gb300 as q4
    N, K = 2048, 16384
    W = synth.normal_rows(5, K, 0, N, 0.02)
    x, xf = x_for(torch.bfloat16, 1, K, seed=7)
    qw = q4.QWeight.from_float(dev_f32(W), compact=True)
    y = q4.gemv(x, qw, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    p, _, z, se = _oracle_compact(W)
    yr, ar = oracle.load().dot_naive(xf, p, se, z, N, K, threads=8)
    compare(y, yr, ar, where="compact gemv long K")


@pytest.mark.parametrize("M,N,K,xdt", [(300, 384, 1024, torch.bfloat16), (17, 160, 2048, torch.float16),
                                       (64, 256, 384, torch.bfloat16), (5, 1000, 128, torch.bfloat16)])
def test_gemm_compact_parity(M, N, K, xdt):
    import weight_only_int4_group_gb300 as q4
    W = synth.normal_rows(M + N, K, 0, N, 0.02)
    x, xf = x_for(xdt, M, K, seed=M + 5)
    qw = q4.QWeight.from_float(dev_f32(W), compact=True)
    p, _, z, se = _oracle_compact(W)
    yr, ar = oracle.load().dot_naive(xf, p, se, z, N, K, threads=8)
    for ydt in (torch.bfloat16, torch.float32):
        y = q4.gemm(x, qw, out_dtype=ydt)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        compare(y, yr, ar, where=f"compact gemm {M}x{N}x{K} y={ydt}")


def test_compact_rejected_by_the_cuda_core_path():
    import weight_only_int4_group_gb300 as q4
    qw = q4.QWeight.from_float(dev_f32(np.zeros((32, 128), np.float32)), compact=True)
    x = torch.zeros((1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.gemv(x, qw, path=q4.PATH_FMA)
    assert ei.value.status == q4.ERR_UNSUPPORTED


def test_layout_mismatch_refused_and_nothing_written():
    """Compact tiles handed over as tiled ones (and the reverse) are refused
    before any launch; the output stays untouched."""
    import weight_only_int4_group_gb300 as q4
    N, K = 200, 1024
    W = synth.normal_rows(12, K, 0, N, 0.02)
    cq = q4.QWeight.from_float(dev_f32(W), compact=True)
    tq = q4.QWeight.from_float(dev_f32(W))
    x = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((2, N), 5.0, device="cuda")
    for bad in (q4.QWeight(cq.data, N, K, compact=False), q4.QWeight(tq.data, N, K, compact=True)):
        for f in (q4.gemv, q4.gemm):
            with pytest.raises(q4.Q4Error) as ei:
                f(x, bad, out=y)
            assert ei.value.status == q4.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 5.0).all())


def test_gemv_compact_fullsize_sampled():
    """28672 x 8192 drawn on the device, M = 1 and M = 16: sampled rows of the
    compact metadata bit-exact and outputs within the tolerance."""
    import weight_only_int4_group_gb300 as q4
    from test_gpu_fullsize import SIGMA, _device_weights
    N, K, seed = 28672, 8192, 151
    w = _device_weights(N, K, seed)
    packed, scale, zero = q4.quantize(w)
    del w
    qw = q4.QWeight(q4.repack_compact(packed, scale, zero, N, K), N, K, compact=True)
    p2, s16, z2 = q4.unpack_compact(qw.data, N, K)
    o = oracle.load()
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 12)]))
    for M in (1, 16):
        xbits = synth.normal_bf16(seed + M, 0, M * K).reshape(M, K)
        y = q4.gemv(dev_bf16_bits(xbits), qw, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        xf = synth.bf16_bits_to_f32(xbits)
        for r in rows:
            Wr = synth.normal_rows(seed, K, int(r), int(r) + 1, SIGMA)
            pr, sr, zr = o.quantize(Wr)
            sr16, zr4 = o.compact_meta(sr, zr)
            se, ze = o.expand_meta(sr16, zr4, K // 128)
            assert np.array_equal(p2[r].cpu().numpy(), pr[0])
            assert np.array_equal(s16[r].cpu().numpy().view(np.uint16), sr16[0])
            assert np.array_equal(z2[r].cpu().numpy(), zr[0])
            yr, ar = o.dot_naive(xf, pr, se, ze, 1, K)
            compare(y[:, r:r + 1], yr, ar, where=f"compact {N}x{K} M={M} row {r}")
