"""Seeded random shapes through both products, against the oracle.

The fixed cases elsewhere pin particular plans; these draw N (often ragged),
K, M, the activation and output types and the weight layout at random from a
fixed seed, so that many plan decisions are crossed -- row-block size, ring
depth, grid sizing, split of K over CTAs or not, the number of contributors
to a row block, the row-split and group-split consumers, the GEMM's token
tile and split plan -- each compared element by element with the oracle's
dequantize-then-dot under the stated tolerance, with the workspace checked
back to zero after every call."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, x_for

pytestmark = pytest.mark.gpu

DT = [torch.bfloat16, torch.float16, torch.float32]


def _draw(rng, product):
    N = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 1200)),
                        int(rng.integers(1200, 6000))]))
    K = 128 * int(rng.choice([1, 2, 3, int(rng.integers(4, 24)), int(rng.integers(24, 72))]))
    if product == "gemv":
        M = int(rng.integers(1, 17))
        xdt = DT[int(rng.integers(0, 3))]  # f32 activations: bf16 hi + lo, any M
    else:
        M = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(40, 400))]))
        xdt = DT[int(rng.integers(0, 2))]
    ydt = DT[int(rng.integers(0, 3))]
    compact = bool(rng.integers(0, 2))
    N = min(N, max(1, int(1.5e9 // (M * K))))  # keeps each oracle product to seconds
    return N, K, M, xdt, ydt, compact


def _run(product, case):
    import weight_only_int4_group_gb300 as q4
    rng = np.random.default_rng(1000 * (product == "gemm") + case)
    N, K, M, xdt, ydt, compact = _draw(rng, product)
    o = oracle.load()
    W = synth.normal_rows(4000 + case, K, 0, N, 0.02)
    p, s, z = o.quantize(W)
    dev = [torch.from_numpy(a).cuda() for a in (p, s, z)]
    if compact:
        qw = q4.QWeight(q4.repack_compact(*dev, N, K), N, K, True)
        s16, z4 = o.compact_meta(s, z)
        s, z = o.expand_meta(s16, z4, K // 128)
    else:
        qw = q4.QWeight(q4.repack(*dev, N, K), N, K)
    x, xf = x_for(xdt, M, K, seed=5000 + case)
    ws = (q4.workspace if product == "gemv" else q4.gemm_workspace)(M, N, K)
    fn = q4.gemv if product == "gemv" else q4.gemm
    y = fn(x, qw, out_dtype=ydt, ws=ws)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    y_ref, absdot = o.dot_naive(xf, p, s, z, N, K, threads=16)
    where = f"{product} case {case}: N={N} K={K} M={M} {xdt}->{ydt} compact={compact}"
    compare(y, y_ref, absdot, where=where)
    if ws is not None:
        assert int(ws.count_nonzero()) == 0, where + ": workspace not left zero"


@pytest.mark.parametrize("case", range(120))
def test_gemv_random_shapes(case):
    _run("gemv", case)


@pytest.mark.parametrize("case", range(40))
def test_gemm_random_shapes(case):
    _run("gemm", case)
