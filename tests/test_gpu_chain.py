"""Launch chains as the benchmark runs them.

Consecutive GEMVs on a stream overlap (programmatic dependent launch): the
next kernel starts copying its weights before the previous one has finished
and reads its activations only after.  These tests make each GEMV read the
previous GEMV's output and check every launch against the oracle applied to
the input that launch actually saw; and they replay the decode-step CUDA graph
exactly as bench.py times it and check sampled rows of its layers."""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import compare

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M", [1, 4, 16])
@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_gemv_chain_feeds_outputs_forward(M, graph):
    """128 GEMVs alternating a 2048 x 4096 and a 4096 x 2048 matrix, each
    reading the previous one's bf16 output, queued back to back with no
    synchronisation (eager, or captured in one CUDA graph).  Every output
    buffer starts filled with a sentinel, so a launch that read its input
    before the previous launch wrote it would be caught."""
    import weight_only_int4_group_gb300 as q4
    o = oracle.load()
    shapes = [(2048, 4096), (4096, 2048)]
    quant, qws = [], []
    for i, (N, K) in enumerate(shapes):
        W = synth.normal_rows(500 + i, K, 0, N, 0.02)
        p, s, z = o.quantize(W)
        quant.append((p, s, z))
        qws.append(q4.QWeight(q4.repack(torch.from_numpy(p).cuda(), torch.from_numpy(s).cuda(),
                                        torch.from_numpy(z).cuda(), N, K), N, K))
    steps = 128
    x0 = torch.from_numpy(synth.normal_bf16(77, 0, M * 4096).view(np.int16)).cuda() \
        .view(torch.bfloat16).view(M, 4096)
    outs = [torch.full((M, shapes[i % 2][0]), 7.0, dtype=torch.bfloat16, device="cuda")
            for i in range(steps)]
    ws = torch.zeros(max(max(q4.gemv_workspace_bytes(M, N, K) for N, K in shapes), 256),
                     dtype=torch.uint8, device="cuda")

    def run():
        x = x0
        for i in range(steps):
            q4.gemv(x, qws[i % 2], out=outs[i], ws=ws)
            x = outs[i]

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()  # first calls outside the capture (plans, kernel attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for t in outs:
            t.fill_(7.0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        for t in outs:
            t.fill_(7.0)
        g.replay()
    else:
        run()
    assert q4.check() == q4.OK
    prev = x0
    for i in range(steps):
        N, K = shapes[i % 2]
        p, s, z = quant[i % 2]
        xf = synth.bf16_bits_to_f32(_bits(prev))
        y_ref, absdot = o.dot_naive(xf, p, s, z, N, K, threads=16)
        compare(outs[i], y_ref, absdot, where=f"step {i}")
        prev = outs[i]
    assert int(ws.count_nonzero()) == 0


def _decode_step_check(M: int, layers: int, check_layers, rows_per_matrix: int = 6):
    """Build the benchmark's decode-step workload, capture and replay its
    graph, and check sampled rows of the given layers against the oracle."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    import weight_only_int4_group_gb300 as q4
    seed = 1000
    work = bench.Decode70B(q4, torch, M, layers, seed=seed)
    work.y.fill_(0)
    g = bench.graph_of(torch, lambda: work.step())
    work.y.fill_(0)
    for _ in range(3):
        g.replay()
    assert q4.check() == q4.OK
    o = oracle.load()
    rng = np.random.default_rng(M * 100 + layers)
    views = work.views()
    for l in check_layers:
        for i, (_, N, K) in enumerate(bench.LAYER_SHAPES):
            xbits = synth.normal_bf16(seed + 7777, work.x_off[l][i], M * K).reshape(M, K)
            xf = synth.bf16_bits_to_f32(xbits)
            y = views[l][i][1]
            rows = np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, rows_per_matrix)]))
            for r in rows:
                Wr = synth.normal_rows(seed + 4 * l + i, K, int(r), int(r) + 1, bench.SIGMA)
                p, s, z = o.quantize(Wr)
                yr, ar = o.dot_naive(xf, p, s, z, 1, K)
                compare(y[:, int(r):int(r) + 1], yr, ar, where=f"layer {l} matrix {i} row {r}")
    del g, work
    torch.cuda.empty_cache()


def test_decode_step_graph_as_timed():
    """The headline workload exactly as timed: 80 layers x 4 GEMVs at M = 1,
    one CUDA graph of 320 overlapping launches sharing one workspace; sampled
    rows of layers 0, 40 and 79 against the oracle."""
    _decode_step_check(1, 80, (0, 40, 79))


def test_decode_step_graph_m8():
    """The same step at M = 8 (the batch-8 kernels), 6 layers."""
    _decode_step_check(8, 6, (0, 3, 5))
