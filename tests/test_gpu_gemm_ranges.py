"""The GEMM's power-of-two normalizations at the edges of their range.

q4_gemm feeds the tensor cores binary16 weights and activations behind exact
powers of two per weight row (from the row's largest group scale) and per
token row (from the row's largest |x|).  These cases hold the parts of that
arithmetic a plain N(0, 1) x N(0, 0.02) product never reaches, each against
the oracle's double-precision dequantize-then-dot, with the relative bound
alone (no absolute allowance, so tiny values are checked as tightly as
large ones):
  * all-zero weight rows and all-zero token rows (their exponent is 0 and
    the result exactly 0);
  * weight rows whose group scales span 2^14, and a row with one outlier
    weight 10^4 among N(0, 0.02) weights (span about 2^18);
  * bf16 token rows scaled by 2^40, 2^-60 and 2^100, far outside binary16;
  * f16 activations up to 60000 next to f16 subnormals.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import dev_bf16_bits, dev_f32

pytestmark = pytest.mark.gpu

N, K = 1024, 1024  # 8 groups per row


def _weights(seed):
    W = synth.normal_rows(seed, K, 0, N, 0.02).astype(np.float64)
    W[5] = 0.0
    W[777] = 0.0
    for r in range(16, 32):  # group g of these rows scaled by 2^(-2g): a 2^14 span
        for g in range(K // 128):
            W[r, 128 * g:128 * (g + 1)] *= 2.0 ** (-2 * g)
    W[40, 300] = 1.0e4  # one outlier: its group's scale is about 2^18 above the others
    return W.astype(np.float32)


def _check(y, W, xf, where):
    o = oracle.load()
    p, s, z = o.quantize(W)
    y_ref, absdot = o.dot_naive(xf, p, s, z, N, K, threads=16)
    g = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - y_ref)
    bound = 1e-3 * absdot
    zero = absdot == 0
    assert np.all(g[zero] == 0.0), f"{where}: a product with no nonzero term is not 0"
    ratio = np.where(zero, 0.0, err / np.where(zero, 1.0, bound))
    worst = float(ratio.max())
    assert worst <= 1.0, f"{where}: worst err / (1e-3 sum|w_hat x|) = {worst:.3g} at " \
                         f"{np.unravel_index(np.argmax(ratio), ratio.shape)}"
    return worst


@pytest.mark.parametrize("M", [40, 200])
def test_gemm_bf16_activation_range(M):
    import weight_only_int4_group_gb300 as q4
    W = _weights(11)
    f = synth.normal(12, 0, M * K).reshape(M, K).astype(np.float64)
    f[3] = 0.0
    f[7] *= 2.0 ** 40
    f[8] *= 2.0 ** -60
    f[9] *= 2.0 ** 100
    f[10, :512] *= 2.0 ** 20  # a token whose two halves differ by 2^20
    bits = synth.to_bf16_bits(f.astype(np.float32))
    x, xf = dev_bf16_bits(bits), synth.bf16_bits_to_f32(bits)
    qw = q4.QWeight.from_float(dev_f32(W))
    y = q4.gemm(x, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    worst = _check(y, W, xf, f"bf16 M={M}")
    assert worst < 2.0 ** -11 / 1e-3 + 0.01, worst


def test_gemm_f16_activation_range():
    import weight_only_int4_group_gb300 as q4
    M = 48
    W = _weights(13)
    f = synth.normal(14, 0, M * K).reshape(M, K)
    f[4] *= 15000.0          # up to about 60000, near the binary16 maximum
    f[5] *= 2.0 ** -20       # binary16 subnormals (exact as given)
    h = np.clip(f, -65000.0, 65000.0).astype(np.float16)
    x, xf = torch.from_numpy(h).cuda(), h.astype(np.float32)
    qw = q4.QWeight.from_float(dev_f32(W))
    y = q4.gemm(x, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    worst = _check(y, W, xf, "f16")
    assert worst < 2.0 ** -11 / 1e-3 + 0.01, worst


def test_gemm_compact_weight_range():
    """The same weight rows in compact tiles (binary16 scales)."""
    import weight_only_int4_group_gb300 as q4
    M = 64
    W = _weights(15)
    bits = synth.normal_bf16(16, 0, M * K).reshape(M, K)
    x, xf = dev_bf16_bits(bits), synth.bf16_bits_to_f32(bits)
    o = oracle.load()
    p, s, z = o.quantize(W)
    dev = [torch.from_numpy(a).cuda() for a in (p, s, z)]
    qw = q4.QWeight(q4.repack_compact(*dev, N, K), N, K, True)
    s16, z4 = o.compact_meta(s, z)
    s2, z2 = o.expand_meta(s16, z4, K // 128)
    y = q4.gemm(x, qw, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    y_ref, absdot = o.dot_naive(xf, p, s2, z2, N, K, threads=16)
    g = y.float().cpu().numpy().astype(np.float64)
    zero = absdot == 0
    assert np.all(g[zero] == 0.0)
    ratio = np.where(zero, 0.0, np.abs(g - y_ref) / np.where(zero, 1.0, 1e-3 * absdot))
    assert float(ratio.max()) < 2.0 ** -11 / 1e-3 + 0.01, float(ratio.max())
