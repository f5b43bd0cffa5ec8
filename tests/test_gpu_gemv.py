"""Decode GEMV (1 <= M <= 16) through the C ABI against the oracle's plain
dequantize-then-dot, element by element, under the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare, dev_f32, oracle_product, x_for

pytestmark = pytest.mark.gpu


def _qweight(W):
    import weight_only_int4_group_gb300 as q4
    return q4.QWeight.from_float(dev_f32(W))


CASES = [
    # (N, K, M): ragged row tiles, a single group, several K slices
    (1, 128, 1), (16, 128, 1), (17, 256, 2), (200, 1024, 1), (200, 1024, 3),
    (64, 2048, 8), (333, 1408, 9), (256, 4096, 16), (48, 8192, 5),
]
DTYPES = [torch.bfloat16, torch.float16, torch.float32]


@pytest.mark.parametrize("N,K,M", CASES)
@pytest.mark.parametrize("xdt", DTYPES, ids=lambda d: str(d).split(".")[-1])
def test_gemv_parity(N, K, M, xdt):
    import weight_only_int4_group_gb300 as q4
    W = synth.normal_rows(5, K, 0, N, 0.02)
    x, xf = x_for(xdt, M, K, seed=N + K + M)
    _, y_ref, absdot = oracle_product(W, xf)
    qw = _qweight(W)
    paths = [q4.PATH_AUTO, q4.PATH_MMA] + ([q4.PATH_FMA] if M == 1 else [])
    for path in paths:
        for ydt in (torch.float32, torch.bfloat16, torch.float16):
            y = q4.gemv(x, qw, out_dtype=ydt, path=path)
            torch.cuda.synchronize()
            assert q4.check() == q4.OK
            compare(y, y_ref, absdot, where=f"path={path} y={ydt}")


def test_gemv_xorshift_4096_f32():
    """The single-GEMV workload: 4096 x 4096, f32 x and y, M = 1, full oracle."""
    import weight_only_int4_group_gb300 as q4
    W, x = synth.xorshift_matrix(4096, 4096)
    _, y_ref, absdot = oracle_product(W, x.reshape(1, -1))
    qw = _qweight(W)
    for path in (q4.PATH_FMA, q4.PATH_MMA):
        y = q4.gemv(dev_f32(x.reshape(1, -1)), qw, out_dtype=torch.float32, path=path)
        stats = compare(y, y_ref, absdot, where=f"xorshift path={path}")
        assert stats["max_err_over_tol"] < 0.05


def test_gemv_outlier_channels():
    """W ~ N(0, 0.02) with 0.1% of input channels multiplied by 20."""
    import weight_only_int4_group_gb300 as q4
    N, K = 512, 4096
    cols = synth.outlier_columns(99, K)
    assert len(cols) == 4
    W = synth.normal_rows(21, K, 0, N, 0.02, cols, 20.0)
    x, xf = x_for(torch.bfloat16, 1, K, seed=4)
    _, y_ref, absdot = oracle_product(W, xf)
    y = q4.gemv(x, _qweight(W), out_dtype=torch.bfloat16)
    compare(y, y_ref, absdot, where="outliers")


def test_gemv_long_runs_per_cta_full_output():
    """M = 1 with many steps per CTA (4096 x 40960: 32 row blocks x 80 steps,
    at least 8 per CTA on a 152-SM part), the case served by the deeper
    copy ring; every output against the oracle, bf16 and f16 activations,
    and bitwise repeatable."""
    import weight_only_int4_group_gb300 as q4
    N, K = 4096, 40960
    W = synth.normal_rows(77, K, 0, N, 0.02)
    qw = _qweight(W)
    o = oracle.load()
    p, s, z = o.quantize(W)
    for xdt in (torch.bfloat16, torch.float16):
        x, xf = x_for(xdt, 1, K, seed=78)
        y_ref, absdot = o.dot_naive(xf, p, s, z, N, K, threads=8)
        y1 = q4.gemv(x, qw, out_dtype=torch.float32)
        y2 = q4.gemv(x, qw, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert q4.check() == q4.OK
        assert torch.equal(y1, y2)
        compare(y1, y_ref, absdot, where=f"long runs x={xdt}")


def test_gemv_deterministic_and_workspace_restored():
    import weight_only_int4_group_gb300 as q4
    N, K, M = 1000, 8192, 4
    W = synth.normal_rows(3, K, 0, N, 0.02)
    x, _ = x_for(torch.bfloat16, M, K, seed=9)
    qw = _qweight(W)
    ws = q4.workspace(M, N, K)
    y1 = q4.gemv(x, qw, out_dtype=torch.float32, ws=ws)
    y2 = q4.gemv(x, qw, out_dtype=torch.float32, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    if ws is not None:
        # counters and partial sums: the whole workspace is back to zero
        assert int(ws.count_nonzero()) == 0


def test_gemv_one_workspace_for_a_decode_layer():
    """A decode layer's pattern with one workspace for every call: shapes with
    different N and K (10240 x 8192, 8192 x 8192, 28672 x 8192, 8192 x
    28672), calls interleaved and repeated; every output equals a call with
    a fresh workspace and the workspace ends zero."""
    import weight_only_int4_group_gb300 as q4
    shapes = [(10240, 8192), (8192, 8192), (28672, 8192), (8192, 28672)]
    qws, xs, refs = [], [], []
    for i, (N, K) in enumerate(shapes):
        w = torch.empty((N, K), dtype=torch.float32, device="cuda")
        synth.dev_normal_f32(w.data_ptr(), N * K, 40 + i, 0, 0.02)
        qws.append(q4.QWeight.from_float(w))
        del w
        xb = torch.empty(K, dtype=torch.int16, device="cuda")
        synth.dev_normal_bf16(xb.data_ptr(), K, 50 + i, 0, 1.0)
        xs.append(xb.view(torch.bfloat16).view(1, K))
        refs.append(q4.gemv(xs[-1], qws[-1], out_dtype=torch.float32))
    need = max(q4.gemv_workspace_bytes(1, N, K) for N, K in shapes)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        for i, (N, K) in enumerate(shapes):
            y = q4.gemv(xs[i], qws[i], out_dtype=torch.float32, ws=ws)
            assert torch.equal(y, refs[i]), (N, K)
    torch.cuda.synchronize()
    assert q4.check() == q4.OK
    assert int(ws.count_nonzero()) == 0


def test_repack_then_gemv_without_sync():
    """The GEMV starts copying weights before it waits for the previous kernel
    on the stream; a repack right before it on the same stream, with no
    synchronisation in between, must still be complete when those copies
    start (the repack kernel does not trigger dependent launches early).
    Each round overwrites the same weight buffer with a different matrix."""
    import weight_only_int4_group_gb300 as q4
    N, K = 4096, 8192
    o = oracle.load()
    x, xf = x_for(torch.bfloat16, 1, K, seed=31)
    qbuf = torch.empty(q4.weight_bytes(N, K), dtype=torch.uint8, device="cuda")
    mats = []
    for r in range(3):
        W = synth.normal_rows(60 + r, K, 0, N, 0.02)
        p, s, z = o.quantize(W)
        mats.append((torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda(),
                     torch.from_numpy(z).cuda(), o.dot_naive(xf, p, s, z, N, K, threads=16)))
    torch.cuda.synchronize()
    ys = []
    for r in range(6):  # no synchronisation until every round is queued
        p, s, z, _ = mats[r % 3]
        q4.repack(p, s, z, N, K, out=qbuf)
        ys.append(q4.gemv(x, q4.QWeight(qbuf, N, K), out_dtype=torch.float32))
    assert q4.check() == q4.OK
    for r, y in enumerate(ys):
        y_ref, absdot = mats[r % 3][3]
        compare(y, y_ref, absdot, where=f"round {r}")


def test_gemv_short_workspace_rejected_and_nothing_written():
    import weight_only_int4_group_gb300 as q4
    N, K, M = 4096, 8192, 1
    if q4.gemv_workspace_bytes(M, N, K) == 0:
        pytest.skip("no split over K for this shape on this device")
    W = synth.normal_rows(1, K, 0, N, 0.02)
    qw = _qweight(W)
    x, _ = x_for(torch.bfloat16, M, K)
    y = torch.full((M, N), 7.0, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q4.Q4Error) as ei:
        q4.gemv(x, qw, out=y, ws=small)
    assert ei.value.status == q4.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_gemv_timeout_path_reports_and_writes_nothing():
    """The producer is told to issue no copy: every consumer wait runs out
    after its bound, the kernel returns without output and q4_check reports
    the timeout.  The context stays usable afterwards."""
    import weight_only_int4_group_gb300 as q4
    N, K, M = 256, 1024, 1
    W = synth.normal_rows(2, K, 0, N, 0.02)
    qw = _qweight(W)
    x, xf = x_for(torch.bfloat16, M, K)
    y = torch.full((M, N), 3.0, device="cuda")
    ws = q4.workspace(M, N, K)
    assert q4.check() == q4.OK
    q4.gemv_timeout_selftest(x, qw, y, ws)
    assert q4.check() == q4.ERR_TIMEOUT
    assert bool((y == 3.0).all())
    assert q4.check() == q4.OK  # the error word was cleared
    # the context still works and the workspace is still usable
    y2 = q4.gemv(x, qw, out_dtype=torch.float32, ws=q4.workspace(M, N, K))
    _, y_ref, absdot = oracle_product(W, xf)
    compare(y2, y_ref, absdot, where="after timeout")
