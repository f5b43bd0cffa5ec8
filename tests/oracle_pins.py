"""Pins: checks that tie the CPU oracle to what the page and the mathematics
fix, independently of the oracle's own code.  Each pin takes an ``Oracle``
and raises AssertionError when the oracle violates it.  The same pins are run
against deliberately broken builds of the oracle to show each planted mistake
is caught (see test_oracle_mutants.py).

Page cited throughout: "Weight quantization" (tirogla.com), sections
"How it works" (formulas) and "Code" (quantize, dot, main).
"""
from __future__ import annotations

import itertools
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = int(v, 0) if v.startswith("0x") else float(v) if "." in v else int(v)
    return out


def _codes(packed: np.ndarray, n_total: int) -> np.ndarray:
    """Unpack with the page's rule: byte idx/2, low nibble = even idx."""
    flat = packed.reshape(-1)
    c = np.empty(n_total, np.int64)
    c[0::2] = flat & 0x0F
    c[1::2] = flat >> 4
    return c


# ----------------------------------------------------------------------------- pins
def pin_page_program(o):
    """The page's own experiment (section "Code", main): the assert holds and
    bits/weight, computed from the page's formula on the oracle's output
    sizes, equals the golden value."""
    gold = read_golden("page_program.txt")
    n = gold["n"]
    r, _ = synth.xorshift_stream(2 * n, gold["seed"])
    w = (np.float32(gold["w_scale"]) * r[:n]).astype(np.float32)
    x = r[n:]
    packed, scale, zero = o.quantize(w)
    dot = o.dot_factored(x, packed, scale, zero, 1, n)[0, 0]
    # exact and scale accumulate in f32 in the page's order
    exact = np.float32(0.0)
    mag = np.float32(0.0)
    for a, b in zip(w, x):
        p = np.float32(a * b)
        exact = np.float32(exact + p)
        mag = np.float32(mag + np.float32(abs(p)))
    assert abs(np.float32(dot - exact)) < np.float32(gold["bound_factor"]) * mag
    bits = (packed.size * 8 + scale.size * 16 + zero.size * 4) / n
    assert bits == gold["bits_per_weight"]
    assert f"{bits:.3f}" == f"{gold['bits_per_weight_printed']:.3f}"


def _integer_group():
    """lo = -5, hi = 10 so that scale = 15/15 = 1 exactly and zero = 5; every
    integer in [-5, 10] then has code w + 5 (closed form)."""
    rng = np.random.default_rng(7)
    v = rng.integers(-5, 11, size=128).astype(np.float32)
    v[0], v[1] = -5.0, 10.0
    return v


def pin_closed_form_integer_group(o):
    """Formulas of "How it works" on a group whose grid is the integers:
    scale 1, zero 5, q = w + 5, w_hat = w exactly, and the byte layout of
    quantize ("low nibble = even index")."""
    v = _integer_group()
    packed, scale, zero = o.quantize(v)
    assert scale[0, 0] == np.float32(1.0)
    assert zero[0, 0] == 5
    q = (v + 5).astype(np.int64)
    expect_bytes = (q[0::2] | (q[1::2] << 4)).astype(np.uint8)
    assert np.array_equal(packed.reshape(-1), expect_bytes)
    wh = o.dequant(packed, scale, zero, 1, 128)
    assert np.array_equal(wh.reshape(-1), v.astype(np.float64))


def pin_round_half_away_codes(o):
    """Ties in w/scale round away from zero (the page's f32::round), and the
    zero is added after rounding: with scale 1 and zero 5, w = 2.5 -> 3+5 = 8
    and w = -2.5 -> -3+5 = 2 (ties-to-even would give 7 and 3; rounding
    w/scale + zero would give 8 and 3)."""
    v = _integer_group()
    v[2], v[3] = 2.5, -2.5
    packed, scale, zero = o.quantize(v)
    assert scale[0, 0] == 1.0 and zero[0, 0] == 5
    c = _codes(packed, 128)
    assert c[2] == 8 and c[3] == 2


def pin_round_half_away_zero(o):
    """lo = -2.5, hi = 12.5: scale = 1 and -lo/scale = 2.5, a tie, so
    zero = round(2.5) = 3 away from zero (2 under ties-to-even)."""
    v = np.zeros(128, np.float32)
    v[:64] = np.linspace(-2.0, 12.0, 64).round()
    v[100], v[101] = -2.5, 12.5
    packed, scale, zero = o.quantize(v)
    assert scale[0, 0] == 1.0
    assert zero[0, 0] == 3


def pin_special_groups(o):
    """Closed forms of the formulas on special groups:
    all-zero -> scale 1 (the page's empty-range branch), zero 0, codes 0;
    all-positive -> zero 0, the maximum maps to 15, 0 would map to 0;
    all-negative -> zero 15, the minimum maps to 0;
    constant c > 0 -> all codes 15; constant c < 0 -> all codes 0."""
    rng = np.random.default_rng(11)
    pos = rng.uniform(0.25, 2.0, 128).astype(np.float32)
    neg = -rng.uniform(0.25, 2.0, 128).astype(np.float32)
    w = np.stack([np.zeros(128, np.float32), pos, neg,
                  np.full(128, 0.7, np.float32), np.full(128, -0.3, np.float32)])
    packed, scale, zero = o.quantize(w)
    c = _codes(packed, w.size).reshape(5, 128)
    assert scale[0, 0] == 1.0 and zero[0, 0] == 0 and not c[0].any()
    assert zero[1, 0] == 0 and c[1][np.argmax(pos)] == 15
    # all-positive: lo clamps to 0, so 15*scale reproduces the maximum to f32 rounding
    assert abs(15.0 * float(scale[1, 0]) - float(pos.max())) <= 2 ** -20 * float(pos.max())
    assert zero[2, 0] == 15 and c[2][np.argmin(neg)] == 0
    assert abs(15.0 * float(scale[2, 0]) + float(neg.min())) <= 2 ** -20 * float(-neg.min())
    assert (c[3] == 15).all() and zero[3, 0] == 0
    assert (c[4] == 0).all() and zero[4, 0] == 15


def _random_groups(rng, N=48, K=512):
    """Groups of varied character: symmetric, skewed, one-signed, with a huge
    outlier, tiny magnitudes, and exact zeros sprinkled in."""
    W = rng.normal(0.0, 0.02, (N, K)).astype(np.float32)
    W[0:4] = np.abs(W[0:4])                       # all >= 0
    W[4:8] = -np.abs(W[4:8])                      # all <= 0
    W[8:12] *= np.float32(1e-30)                  # tiny
    W[12:16, ::37] *= np.float32(100.0)           # outliers
    W[16:20] += np.float32(0.05)                  # skewed
    W[rng.random((N, K)) < 0.03] = 0.0            # exact zeros
    return W


def pin_zero_exact(o):
    """The range is widened to contain 0 ("keep 0 exactly representable"),
    so every w == 0 reconstructs to exactly 0, and 0 <= zero <= 15."""
    rng = np.random.default_rng(3)
    W = _random_groups(rng)
    N, K = W.shape
    packed, scale, zero = o.quantize(W)
    wh = o.dequant(packed, scale, zero, N, K)
    assert (zero <= 15).all()
    assert (wh[W == 0] == 0.0).all()


def pin_half_step(o):
    """Rounding error is at most half a step: |w - w_hat| <= scale/2 for every
    element, the clamped extremes included (lo >= -zero*s - s/2 since zero
    rounds -lo/s; hi <= (15-zero)*s + s/2 since hi - lo = 15 s).  Checked in
    double with a few f32 ulps of slack for the rounding of s itself."""
    rng = np.random.default_rng(5)
    W = _random_groups(rng)
    N, K = W.shape
    packed, scale, zero = o.quantize(W)
    wh = o.dequant(packed, scale, zero, N, K)
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    err = np.abs(W.astype(np.float64) - wh)
    assert (err <= 0.5 * s * (1 + 2 ** -16) + 16 * np.abs(W) * 2.0 ** -24).all()


def pin_brute_force_tiny(o):
    """Brute force over every group of size 2 and 3 on a grid of values
    (multiples of 1/8 in [-1, 1]): the chosen code is a nearest point of the
    group's 16-point grid (q - zero)*scale, up to the f32 rounding of w/scale,
    scale spans the widened range (15*scale == hi - lo to f32 rounding) and
    zero is the nearest integer to -lo/scale."""
    vals = np.arange(-8, 9, dtype=np.float32) / np.float32(8.0)
    for G in (2, 3):
        groups = np.array(list(itertools.product(vals, repeat=G)), np.float32)
        if G == 3:
            groups = groups[::5]
        W = groups.reshape(1, -1)
        if W.shape[1] % 2:
            W = W[:, :-G]
        ng = W.shape[1] // G
        packed, scale, zero = o.quantize(W, group=G)
        c = _codes(packed, W.shape[1]).reshape(ng, G)
        Wg = W.reshape(ng, G).astype(np.float64)
        s = scale.reshape(ng).astype(np.float64)
        z = zero.reshape(ng).astype(np.float64)
        lo = np.minimum(Wg.min(1), 0.0)
        hi = np.maximum(Wg.max(1), 0.0)
        empty = hi == lo
        assert (s[empty] == 1.0).all()
        ne = ~empty
        assert np.allclose(15.0 * s[ne], (hi - lo)[ne], rtol=2 ** -22, atol=0)
        assert (np.abs(z[ne] - (-lo[ne] / s[ne])) <= 0.5 + 1e-6).all()
        grid = (np.arange(16)[None, None, :] - z[:, None, None]) * s[:, None, None]
        dist = np.abs(Wg[:, :, None] - grid)
        chosen = np.take_along_axis(dist, c[:, :, None], axis=2)[:, :, 0]
        # a near-tie may go either way because w/scale is an f32 quotient
        slack = 2.0 ** -20 * s[:, None] + 2.0 ** -22 * np.abs(Wg)
        assert (chosen <= dist.min(axis=2) + slack).all()


def pin_dot_definition(o):
    """The plain product against numpy's matmul of the dequantized matrix
    (a library routine standing in for the definition sum_k w_hat*x), on a
    non-square shape so that a transposed operand cannot pass."""
    rng = np.random.default_rng(9)
    for (N, K, M) in ((40, 384, 3), (256, 256, 2)):
        W = rng.normal(0, 0.02, (N, K)).astype(np.float32)
        X = rng.normal(0, 1, (M, K)).astype(np.float32)
        packed, scale, zero = o.quantize(W)
        wh = o.dequant(packed, scale, zero, N, K)
        y, a = o.dot_naive(X, packed, scale, zero, N, K)
        ref = X.astype(np.float64) @ wh.T
        aref = np.abs(X.astype(np.float64)) @ np.abs(wh).T
        assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(a, aref, rtol=1e-12, atol=1e-12)
        # sub-range of rows gives the same numbers
        y2, _ = o.dot_naive(X, packed, scale, zero, N, K, 5, 17)
        assert np.array_equal(y2, y[:, 5:17])


def pin_factored_identity(o):
    """The factored group dot scale*(sum q*x - zero*sum x) ("How it works")
    equals the naive dequantize-then-dot, up to f32 accumulation error."""
    rng = np.random.default_rng(13)
    N, K, M = 64, 1024, 3
    W = _random_groups(rng, N, K)
    X = rng.normal(0, 1, (M, K)).astype(np.float32)
    packed, scale, zero = o.quantize(W)
    yf = o.dot_factored(X, packed, scale, zero, N, K).astype(np.float64)
    yn, a = o.dot_naive(X, packed, scale, zero, N, K)
    assert (np.abs(yf - yn) <= 1e-5 * a + 1e-30).all()


def pin_xsum(o):
    """Activation group sums against numpy's sum."""
    rng = np.random.default_rng(17)
    X = rng.normal(0, 1, (3, 640)).astype(np.float32)
    ref = X.astype(np.float64).reshape(3, 5, 128).sum(-1)
    assert np.allclose(o.xsum(X), ref, rtol=1e-13, atol=1e-13)


def pin_matrix_bound(o, N: int = 1024, K: int = 4096):
    """The page's bound |err| < 0.02*sum|w*x| holds for every row of the
    xorshift-drawn matrix (w = 0.02*U(-1,1) row-major, then x = U(-1,1)),
    with the exact product taken on the unquantized weights in double."""
    W, x = synth.xorshift_matrix(N, K)
    packed, scale, zero = o.quantize(W)
    y, _ = o.dot_naive(x, packed, scale, zero, N, K, threads=4)
    exact = W.astype(np.float64) @ x.astype(np.float64)
    mag = np.abs(W.astype(np.float64)) @ np.abs(x.astype(np.float64))
    assert (np.abs(y[0] - exact) < 0.02 * mag).all()



# --------------------------------------------------------- symmetric variant
# Page cited: "Quantization" (hritesh-sonawane.github.io notes), sections
# "How it really works" (scale = max|x| / (2^(b-1) - 1), q = clamp(round(x /
# scale)), x_hat = q * scale) and "Code" (int_quant and its printed table).

def _sym_codes(o, W, group=128):
    W = np.atleast_2d(np.asarray(W, np.float32))
    packed, scale, zero = o.quantize(W, group=group, symmetric=True)
    c = _codes(packed, W.size).reshape(W.shape)
    return c, scale, zero


def pin_sym_page_table(o):
    """The INT4 rows of the page's printed error table (per tensor, per
    channel, group 128, group 32), reproduced on the page's own synthetic
    matrix to the printed precision."""
    gold = read_golden("page_int4_error_table.txt")
    R, C = gold["rows"], gold["cols"]
    w = synth.row_scaled_outliers(R, C, gold["seed"])
    wf = w.astype(np.float32)
    for key, shape, group in (("tensor", (1, R * C), R * C), ("channel", (R, C), C),
                              ("g128", (R, C), 128), ("g32", (R, C), 32)):
        packed, scale, zero = o.quantize(wf.reshape(shape), group=group, symmetric=True)
        wh = o.dequant(packed, scale, zero, shape[0], shape[1], group=group).reshape(R, C)
        sig = float((w * w).sum())
        err = float(((w - wh) ** 2).sum())
        assert f"{10 * np.log10(sig / err):.1f}" == f"{gold[key + '_sqnr_db']:.1f}", key
        assert f"{100 * np.sqrt(err / sig):.2f}" == f"{gold[key + '_rel_pct']:.2f}", key


def pin_sym_ties_to_even(o):
    """With max|w| = 7 the scale is exactly 1, so w / scale = w: the halves
    2.5, -2.5, 3.5, -0.5, 6.5 round to the even neighbours 2, -2, 4, 0, 6
    (Python's round and torch.round, which both pages use); stored codes are
    q + 8 with zero 8."""
    v = np.zeros(128, np.float32)
    v[0] = 7.0
    v[1:6] = [2.5, -2.5, 3.5, -0.5, 6.5]
    v[6:10] = [1.0, -7.0, -3.0, 0.25]
    c, scale, zero = _sym_codes(o, v)
    assert scale[0, 0] == np.float32(1.0) and zero[0, 0] == 8
    assert list(c[0, :10] - 8) == [7, 2, -2, 4, 0, 6, 1, -7, -3, 0]


def pin_sym_special_groups(o):
    """Closed forms: an all-zero group has scale 1 (the page's "or 1.0") and
    codes 8; a constant group c has scale |c|/7 and q = +-7; the largest
    magnitude always maps to +-7; a group whose max|w|/7 underflows to 0 gets
    scale 1 as well."""
    tiny = np.float32(np.ldexp(1.0, -149))
    rng = np.random.default_rng(21)
    mixed = rng.normal(0, 0.02, 128).astype(np.float32)
    W = np.stack([np.zeros(128, np.float32), np.full(128, 0.7, np.float32),
                  np.full(128, -0.3, np.float32), mixed, np.full(128, tiny, np.float32)])
    c, scale, zero = _sym_codes(o, W)
    q = c.astype(np.int64) - 8
    assert (zero == 8).all()
    assert scale[0, 0] == 1.0 and (q[0] == 0).all()
    assert scale[1, 0] == np.float32(0.7) / np.float32(7.0) and (q[1] == 7).all()
    assert scale[2, 0] == np.float32(0.3) / np.float32(7.0) and (q[2] == -7).all()
    i = int(np.argmax(np.abs(mixed)))
    assert q[3, i] == (7 if mixed[i] > 0 else -7)
    assert abs(7.0 * float(scale[3, 0]) - abs(float(mixed[i]))) <= 2 ** -21 * abs(float(mixed[i]))
    assert scale[4, 0] == 1.0 and (q[4] == 0).all()


def pin_sym_half_step_and_nearest(o):
    """|w - w_hat| <= scale/2 for every element (no clamping occurs since
    |w / scale| <= 7), w == 0 reconstructs to 0, and each code is a nearest
    point of the grid {-8..7} * scale up to the f32 rounding of w / scale."""
    rng = np.random.default_rng(23)
    W = _random_groups(rng)
    N, K = W.shape
    c, scale, zero = _sym_codes(o, W)
    wh = o.dequant(*o.quantize(W, symmetric=True), N, K)
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    Wd = W.astype(np.float64)
    assert (np.abs(Wd - wh) <= 0.5 * s * (1 + 2 ** -16) + 16 * np.abs(Wd) * 2.0 ** -24).all()
    assert (wh[W == 0] == 0.0).all()
    grid = np.arange(-8, 8, dtype=np.float64)
    dist = np.abs(Wd[:, :, None] - grid[None, None, :] * s[:, :, None])
    chosen = np.take_along_axis(dist, (c.astype(np.int64))[:, :, None], axis=2)[:, :, 0]
    assert (chosen <= dist.min(axis=2) + 2.0 ** -20 * s + 2.0 ** -22 * np.abs(Wd)).all()



# ------------------------------------------------- compact metadata (fp16, 4-bit)
# Page cited: "Weight quantization", section "Code" (bits per weight with
# 16-bit scales and 4-bit zeros), "Complexity and constants" (fp16 scale +
# 4-bit zero), "Implementation notes" (scales in fp16/bf16).

def pin_f16_rounding_library(o):
    """binary16 rounding against numpy's float16 conversion (IEEE round to
    nearest even): random finite f32 bit patterns over the whole range, every
    midpoint between neighbouring binary16 values (ties), the overflow edge;
    and the exact widening of all 63488 finite binary16 patterns."""
    rng = np.random.default_rng(31)
    bits = rng.integers(0, 0xFF000000, 200_000, dtype=np.uint64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]
    # keep most samples near binary16's range, where rounding is not trivial
    near = (rng.integers(0x30000000, 0x48000000, 200_000, dtype=np.uint64).astype(np.uint32)
            | (rng.integers(0, 2, 200_000, dtype=np.uint64).astype(np.uint32) << 31))
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)  # finite, non-negative
    lo = h[:-1].view(np.float16).astype(np.float64)
    hi = h[1:].view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)                     # exact in f32
    mids = mids[mids.astype(np.float64) == (lo + hi) / 2]
    edge = np.array([65504.0, 65519.996, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                     6.1035156e-05, 6.0975552e-05, 0.0, -0.0], np.float32)
    v = np.concatenate([bits.view(np.float32), near.view(np.float32), mids, -mids, edge])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(o.f16_bits(v), ref)
    allh = np.concatenate([h, h | np.uint16(0x8000)])
    assert np.array_equal(o.f16_values(allh).view(np.uint32),
                          allh.view(np.float16).astype(np.float32).view(np.uint32))


def pin_compact_meta_layout(o):
    """Compacting keeps every zero (two per byte, even group in the low
    nibble, an odd count padded with a zero nibble) and stores each scale as
    its nearest-even binary16 (numpy's conversion); expanding widens it back
    exactly."""
    rng = np.random.default_rng(37)
    for NG in (1, 2, 7, 64):
        scale = rng.uniform(1e-4, 0.05, (5, NG)).astype(np.float32)
        zero = rng.integers(0, 16, (5, NG)).astype(np.uint8)
        s16, z4 = o.compact_meta(scale, zero)
        assert np.array_equal(s16, scale.astype(np.float16).view(np.uint16))
        zpad = np.concatenate([zero, np.zeros((5, NG % 2), np.uint8)], axis=1)
        assert np.array_equal(z4, (zpad[:, 0::2] | (zpad[:, 1::2] << 4)).astype(np.uint8))
        s2, z2 = o.expand_meta(s16, z4, NG)
        assert np.array_equal(z2, zero)
        assert np.array_equal(s2, scale.astype(np.float16).astype(np.float32))


def pin_compact_bits_per_weight(o):
    """The page's program counts 16-bit scales and 4-bit zeros: on its n =
    4096 weights the compact arrays come to exactly its 4.15625 bits/weight."""
    gold = read_golden("page_program.txt")
    w, _ = synth.page_program(gold["n"])
    packed, scale, zero = o.quantize(w)
    s16, z4 = o.compact_meta(scale, zero)
    bits = (packed.size * 8 + s16.size * 16 + z4.size * 8) / gold["n"]
    assert bits == gold["bits_per_weight"]


def pin_compact_error_bound(o):
    """With the scale stored as binary16 (relative error at most 2^-11 in its
    normal range) the reconstruction stays within half a step plus the
    scale's rounding times the largest |q - zero| (15)."""
    rng = np.random.default_rng(41)
    W = rng.normal(0, 0.02, (32, 1024)).astype(np.float32)
    W[0:4, ::37] *= np.float32(20.0)
    N, K = W.shape
    packed, scale, zero = o.quantize(W)
    s16, z4 = o.compact_meta(scale, zero)
    sc, zc = o.expand_meta(s16, z4, K // 128)
    wh = o.dequant(packed, sc, zc, N, K)
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    ds = np.repeat(np.abs(sc.astype(np.float64) - scale.astype(np.float64)), 128, axis=1)
    assert (np.abs(scale - sc) <= 2.0 ** -11 * scale).all()
    err = np.abs(W.astype(np.float64) - wh)
    assert (err <= 0.5 * s * (1 + 2 ** -16) + 15 * ds + 16 * np.abs(W) * 2.0 ** -24).all()


ALL_PINS = [
    pin_page_program,
    pin_closed_form_integer_group,
    pin_round_half_away_codes,
    pin_round_half_away_zero,
    pin_special_groups,
    pin_zero_exact,
    pin_half_step,
    pin_brute_force_tiny,
    pin_dot_definition,
    pin_factored_identity,
    pin_xsum,
    pin_matrix_bound,
    pin_sym_page_table,
    pin_sym_ties_to_even,
    pin_sym_special_groups,
    pin_sym_half_step_and_nearest,
    pin_f16_rounding_library,
    pin_compact_meta_layout,
    pin_compact_bits_per_weight,
    pin_compact_error_bound,
]
