"""GPU quantize/pack against the oracle: codes, scales and zeros bit-exact;
repack/unpack round trip; activation group sums."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import dev_f32

pytestmark = pytest.mark.gpu


def _edge_matrix(N, K, seed):
    rng = np.random.default_rng(seed)
    W = rng.normal(0, 0.02, (N, K)).astype(np.float32)
    if N >= 12:
        W[0] = 0.0                                       # all-zero groups (empty range)
        W[1] = np.abs(W[1])                              # all >= 0
        W[2] = -np.abs(W[2])                             # all <= 0
        W[3] = np.float32(0.37)                          # constant > 0
        W[4] = np.float32(-0.11)                         # constant < 0
        W[5] = rng.integers(-5, 11, K).astype(np.float32)  # scale 1, zero 5, exact ties below
        W[5, ::128] = -5.0
        W[5, 1::128] = 10.0
        W[5, 2::7] = 2.5                                 # ties of w/scale
        W[5, 3::7] = -2.5
        W[6] *= np.float32(1e-30)                        # subnormal-range scales
        W[7, ::37] *= np.float32(100.0)                  # outliers
        W[8] += np.float32(0.05)                         # skewed
        W[9, ::128] = -2.5                               # zero tie: -lo/scale = 2.5
        W[9, 1::128] = 12.5
        W[9, 2::128] = 0.0
        W[10][rng.random(K) < 0.2] = 0.0                 # exact zeros
        W[11] = -0.0                                     # negative zeros
    if N >= 14:
        W[12] = np.float32(np.ldexp(3.0, -149))          # subnormal weights, subnormal scale
        W[12, 1::5] = np.float32(np.ldexp(-7.0, -149))
        W[13] = np.float32(np.ldexp(40.0, -149))         # one-signed subnormal group
        # (a range below 15 x the smallest subnormal would make the scale 0:
        # outside the contract, like non-finite weights)
    return W


SHAPES = [(1, 128), (2, 256), (12, 128), (14, 256), (200, 1024), (33, 4096), (16, 11008)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_bit_exact(N, K):
    W = _edge_matrix(N, K, seed=N * 7 + K)
    import weight_only_int4_group_gb300 as q4
    p, s, z = q4.quantize(dev_f32(W))
    torch.cuda.synchronize()
    po, so, zo = oracle.load().quantize(W)
    assert np.array_equal(p.cpu().numpy(), po)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zo)


def test_quantize_near_tie_quotients():
    """Weights whose quotient w / scale lies within a few ulps of a rounding
    boundary n + 1/2 (both sides): the codes must follow the IEEE f32
    quotient exactly."""
    import weight_only_int4_group_gb300 as q4
    rng = np.random.default_rng(17)
    N, K = 64, 1024
    W = np.empty((N, K), dtype=np.float32)
    for r in range(N):
        for g in range(K // 128):
            lo = -np.float32(rng.uniform(0.01, 1.0))
            hi = np.float32(rng.uniform(0.01, 1.0))
            s = np.float32(np.float32(hi - lo) / np.float32(15.0))
            n = rng.integers(-7, 7, 126).astype(np.float32)
            w = np.float32((n + np.float32(0.5)) * s)
            steps = rng.integers(-3, 4, 126)
            for i, k in enumerate(steps):  # a few ulps either way
                for _ in range(abs(int(k))):
                    w[i] = np.nextafter(w[i], np.float32(np.inf if k > 0 else -np.inf))
            w = np.clip(w, lo, hi)
            W[r, g * 128:(g + 1) * 128] = np.concatenate([[lo, hi], w])
    p, s_, z = q4.quantize(dev_f32(W))
    po, so, zo = oracle.load().quantize(W)
    assert np.array_equal(s_.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zo)
    assert np.array_equal(p.cpu().numpy(), po)


def test_quantize_page_program():
    import weight_only_int4_group_gb300 as q4
    w, _ = synth.page_program()
    p, s, z = q4.quantize(dev_f32(w.reshape(1, -1)))
    po, so, zo = oracle.load().quantize(w)
    assert np.array_equal(p.cpu().numpy(), po)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zo)


def test_quantize_xorshift_4096_full():
    """The whole 4096 x 4096 single-GEMV matrix (w = 0.02*U(-1,1), xorshift)."""
    import weight_only_int4_group_gb300 as q4
    W, _ = synth.xorshift_matrix(4096, 4096)
    p, s, z = q4.quantize(dev_f32(W))
    po, so, zo = oracle.load().quantize(W)
    assert np.array_equal(p.cpu().numpy(), po)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), so.view(np.uint32))
    assert np.array_equal(z.cpu().numpy(), zo)


@pytest.mark.parametrize("N,K", [(1, 128), (15, 256), (16, 128), (17, 384), (200, 1024)])
def test_repack_unpack_round_trip(N, K):
    import weight_only_int4_group_gb300 as q4
    rng = np.random.default_rng(N + K)
    packed = torch.from_numpy(rng.integers(0, 256, (N, K // 2), dtype=np.uint8)).cuda()
    scale = torch.from_numpy(rng.normal(0, 1, (N, K // 128)).astype(np.float32)).cuda()
    zero = torch.from_numpy(rng.integers(0, 16, (N, K // 128), dtype=np.uint8)).cuda()
    qw = q4.repack(packed, scale, zero, N, K)
    assert qw.numel() == q4.weight_bytes(N, K)
    p2, s2, z2 = q4.unpack(qw, N, K)
    assert torch.equal(p2, packed)
    assert torch.equal(s2.view(torch.int32), scale.view(torch.int32))
    assert torch.equal(z2, zero)
    # padded rows of the last tile are zero
    ntiles = (N + 15) // 16
    if N % 16:
        # the last row tile's tiles, found by the documented tile order
        NG = K // 128
        tiles = qw.view(ntiles * NG, 1104).cpu().numpy()
        t = np.stack([tiles[_tile_number(ntiles - 1, g, ntiles, NG)] for g in range(NG)])
        # scale pairs of rows >= N (within the tile) are 0.0
        sp = t[:, 1024:1088].view(np.float32).reshape(NG, 8, 2)
        for r in range(N % 16, 16):
            assert (sp[:, r % 8, r // 8] == 0).all()


def test_repack_field_layout():
    """One code placed at a known (row, k) lands in the nibble field the
    header documents."""
    import weight_only_int4_group_gb300 as q4
    N, K = 16, 128
    for (row, k, lane, chunk, word, shift) in [
            (0, 0, 0, 0, 0, 0), (0, 1, 0, 0, 0, 16), (8, 0, 0, 0, 0, 4), (8, 1, 0, 0, 0, 20),
            (8, 8, 0, 0, 0, 8), (8, 9, 0, 0, 0, 24), (0, 8, 0, 0, 0, 12), (0, 9, 0, 0, 0, 28),
            (3, 6, 15, 0, 0, 0), (3, 16 * 5 + 7, 15, 1, 1, 16), (11, 16 * 7 + 15, 15, 1, 3, 24)]:
        packed = np.zeros((N, K // 2), np.uint8)
        packed[row, k // 2] = (9 << 4) if k % 2 else 9
        qw = q4.repack(torch.from_numpy(packed).cuda(), torch.zeros((N, 1), device="cuda"),
                       torch.zeros((N, 1), dtype=torch.uint8, device="cuda"), N, K).cpu().numpy()
        words = qw[:1024].view(np.uint32).reshape(2, 32, 4)
        expect = np.zeros_like(words)
        expect[chunk, lane, word] = 9 << shift
        assert np.array_equal(words, expect), (row, k)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_xsum(dtype):
    import weight_only_int4_group_gb300 as q4
    from gpu_helpers import x_for
    x, xf = x_for(dtype, 5, 1024, seed=3)
    got = q4.xsum(x).cpu().numpy().astype(np.float64)
    ref = oracle.load().xsum(xf)
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-4)


def _tile_number(rt, g, T, NG):
    """The tile order include/q4.h states (restated independently here)."""
    b, s = rt // 8, g // 4
    nb, ns = min(8, T - 8 * b), min(4, NG - 4 * s)
    return 8 * NG * b + nb * 4 * s + (rt - 8 * b) * ns + (g - 4 * s)


@pytest.mark.parametrize("compact", [False, True])
@pytest.mark.parametrize("N,K", [(300, 1152), (128, 512), (2000, 640)])
def test_repack_tile_order(N, K, compact):
    """Each tile's scales name its (row tile, group): every row of row tile
    rt has scale 1 + rt + 128 g in group g (an integer below 2048, exact in
    binary16), and every tile sits where the documented order puts it;
    ragged last block (300 rows: 19 tiles) and last step (9 or 5 groups)."""
    import weight_only_int4_group_gb300 as q4
    T, NG = (N + 15) // 16, K // 128
    packed = torch.zeros((N, K // 2), dtype=torch.uint8, device="cuda")
    rows = torch.arange(N, dtype=torch.float32).view(N, 1)
    groups = torch.arange(NG, dtype=torch.float32).view(1, NG)
    scale = (rows // 16 + 128.0 * groups + 1.0).cuda()
    zero = torch.zeros((N, NG), dtype=torch.uint8, device="cuda")
    rep = q4.repack_compact if compact else q4.repack
    tb = 1072 if compact else 1104
    qw = rep(packed, scale, zero, N, K).cpu().numpy()
    assert qw.size == T * NG * tb
    seen = set()
    for t in range(T * NG):
        tile = qw[t * tb:(t + 1) * tb]
        if compact:
            s0 = float(tile[1024:1026].view(np.float16)[0])
        else:
            s0 = float(tile[1024:1028].view(np.float32)[0])
        rt, g = int(s0 - 1) % 128, int(s0 - 1) // 128
        assert _tile_number(rt, g, T, NG) == t, (t, rt, g)
        seen.add((rt, g))
    assert len(seen) == T * NG
