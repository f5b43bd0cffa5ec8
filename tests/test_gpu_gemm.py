"""W4A16 GEMM (tcgen05, binary16 operands) through the C ABI against the
oracle's plain dequantize-then-dot, element by element, under the stated
tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_f32, oracle_product, x_for

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
    for ydt in (torch.bfloat16, torch.float16, torch.float32):
        y = q4.gemm(x, qw, out_dtype=ydt)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        compare(y, y_ref, absdot, where=f"gemm {M}x{N}x{K} y={ydt}")


@pytest.mark.parametrize("K", [128, 256, 384, 512])
@pytest.mark.parametrize("dist", ["normal", "outlier"])
def test_gemm_small_k_many_rows(K, dist):
    """Short K (one to four groups), where a single weight's error is not
    averaged away: 4096 rows x 256 tokens, three seeds, plain N(0, 0.02)
    weights and weights with one input channel scaled x20 (most weights of
    that group then quantize to the zero point).  f32 output, so the
    comparison sees the product itself.  Each weight enters the tensor cores
    rounded once to binary16 (relative error at most 2^-11), so no element
    may use more than 2^-11 / 1e-3 = 0.49 of the tolerance, whatever the
    signs line up to."""
    import weight_only_int4_group_gb300 as q4
    N, M = 4096, 256
    worst = 0.0
    for seed in range(3):
        cols = np.array([(seed * 37 + 11) % K], np.int32) if dist == "outlier" else None
        W = synth.normal_rows(seed + 100 * K, K, 0, N, 0.02, cols, 20.0)
        x, xf = x_for(torch.bfloat16, M, K, seed=seed + 7)
        _, y_ref, absdot = oracle_product(W, xf, threads=16)
        y = q4.gemm(x, q4.QWeight.from_float(dev_f32(W)), out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        worst = max(worst, compare(y, y_ref, absdot, where=f"K={K} {dist} seed {seed}")
                    ["max_err_over_tol"])
    # the worst case of one binary16 rounding per term, plus f32 accumulation
    assert worst < 2.0 ** -11 / 1e-3 + 0.01, worst


@pytest.mark.parametrize("M", [1, 9, 16, 17, 32, 48, 64, 100, 128, 129, 255])
def test_gemm_small_m(M):
    """q4_gemm accepts any M >= 1; the token tile (16, 32, 64 or 128 rows) is
    the smallest that covers M, with a ragged last tile; few tiles split
    their groups over several CTAs."""
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


@pytest.mark.parametrize("N", [1, 15, 100, 130])
def test_gemm_ragged_n(N):
    """Output sizes that are not multiples of 16 or 128."""
    import weight_only_int4_group_gb300 as q4
    M, K = 40, 1024
    W = synth.normal_rows(N + 5, K, 0, N, 0.02)
    x, xf = x_for(torch.bfloat16, M, K, seed=N)
    _, y_ref, absdot = oracle_product(W, xf)
    y = q4.gemm(x, q4.QWeight.from_float(dev_f32(W)), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    compare(y, y_ref, absdot, where=f"gemm N={N}")


def test_gemm_split_deterministic_and_workspace_cleared():
    """Few tokens on a long K: the groups of each tile are spread over
    several CTAs.  Results are bitwise repeatable, and a completed call
    leaves the whole workspace zero."""
    import weight_only_int4_group_gb300 as q4
    M, N, K = 24, 1024, 16384
    need = q4.gemm_workspace_bytes(M, N, K)
    assert need > 0
    W = synth.normal_rows(8, K, 0, N, 0.02)
    x, xf = x_for(torch.bfloat16, M, K, seed=9)
    qw = q4.QWeight.from_float(dev_f32(W))
    ws = q4.gemm_workspace(M, N, K)
    y1 = q4.gemm(x, qw, out_dtype=torch.float32, ws=ws)
    y2 = q4.gemm(x, qw, out_dtype=torch.float32, ws=ws)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    assert torch.equal(y1, y2)
    assert int(ws.count_nonzero()) == 0
    _, y_ref, absdot = oracle_product(W, xf)
    compare(y1, y_ref, absdot, where="split")


def test_one_workspace_serves_every_shape():
    """One zero-filled buffer, the largest any call needs, shared by GEMVs and
    GEMMs of different N, M and K on one stream: every result equals the call
    with a fresh workspace and the buffer ends zero."""
    import weight_only_int4_group_gb300 as q4
    shapes = [(3000, 4096), (8192, 2048), (1000, 8192), (4096, 4096)]
    qws = {s: q4.QWeight.from_float(dev_f32(synth.normal_rows(sum(s), s[1], 0, s[0], 0.02)))
           for s in shapes}
    calls = [("gemv", 1), ("gemv", 4), ("gemv", 16), ("gemm", 24), ("gemm", 64)]
    need = max(max(q4.gemv_workspace_bytes(16, N, K), q4.gemm_workspace_bytes(64, N, K))
               for N, K in shapes)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for (N, K) in shapes:
            for kind, M in calls:
                x, _ = x_for(torch.bfloat16, M, K, seed=M + K + rep)
                f = q4.gemv if kind == "gemv" else q4.gemm
                ref = f(x, qws[(N, K)], out_dtype=torch.float32)  # fresh workspace
                y = f(x, qws[(N, K)], out_dtype=torch.float32, ws=ws)
                assert torch.equal(y, ref), (kind, M, N, K)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    assert int(ws.count_nonzero()) == 0


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
    # a buffer declared with the wrong layout is refused before any launch
    xb = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    bad = q4.QWeight(qw.data, 32, 128, compact=True)
    with pytest.raises(q4.Q4Error) as ei:
        q4.gemm(xb, bad)
    assert ei.value.status == q4.ERR_INVALID_ARG


@pytest.mark.parametrize("M", [8, 300])
def test_gemm_timeout_path_reports_and_writes_nothing(M):
    """The weight copies are switched off: the operand builders' waits run
    out after their bound, every role stops, tensor memory is freed and the
    kernel returns without output; q4_check reports the timeout.  A normal
    call afterwards (same tensor memory, same SMs) matches the oracle."""
    import weight_only_int4_group_gb300 as q4
    N, K = 256, 1024
    W = synth.normal_rows(4, K, 0, N, 0.02)
    qw = q4.QWeight.from_float(dev_f32(W))
    x, xf = x_for(torch.bfloat16, M, K, seed=6)
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    ws = q4.gemm_workspace(M, N, K)
    assert q4.check() == q4.OK
    q4.gemm_timeout_selftest(x, qw, y, ws)
    assert q4.check() == q4.ERR_TIMEOUT
    assert bool((y == 3.0).all())
    assert q4.check() == q4.OK  # the error word was cleared
    _, y_ref, absdot = oracle_product(W, xf)
    y2 = q4.gemm(x, qw, out_dtype=torch.float32, ws=q4.gemm_workspace(M, N, K))
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    compare(y2, y_ref, absdot, where="after timeout")


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


@pytest.mark.parametrize("xdt,compact", [(torch.bfloat16, False), (torch.float16, True)])
def test_gemm_256_token_tiles(xdt, compact):
    """A shape whose 256-token tiles alone give every SM of a 152-SM GPU
    eight or more (3 token tiles x 407 row blocks = 1221), so the GEMM takes
    256-token tiles with one tensor-memory accumulator per tile: ragged in
    both M (513 = 2 x 256 + 1) and N, every element against the oracle."""
    import weight_only_int4_group_gb300 as q4
    M, N, K = 513, 407 * 128 - 5, 128
    W = synth.normal_rows(77, K, 0, N, 0.02)
    x, xf = x_for(xdt, M, K, seed=78)
    o = oracle.load()
    p, s, z = o.quantize(W)
    dev = [torch.from_numpy(a).cuda() for a in (p, s, z)]
    if compact:
        qw = q4.QWeight(q4.repack_compact(*dev, N, K), N, K, True)
        s16, z4 = o.compact_meta(s, z)
        s, z = o.expand_meta(s16, z4, K // 128)
    else:
        qw = q4.QWeight(q4.repack(*dev, N, K), N, K)
    ws = q4.gemm_workspace(M, N, K)
    y = q4.gemm(x, qw, out_dtype=torch.bfloat16, ws=ws)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    assert int(ws.count_nonzero()) == 0
    y_ref, absdot = o.dot_naive(xf, p, s, z, N, K, threads=16)
    compare(y, y_ref, absdot, where=f"256-token tiles {xdt} compact={compact}")
