"""The benchmark's multi-process host logic on CPU (gloo, world size 2):
every replica's time reduces to the slowest one on all ranks, and the
whole-job value counts every replica's bytes over that time.  No GPU: the
replicas share nothing on the data path, so this is the only exchange."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, ws: int, port: int, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        times = [0.004, 0.0075]  # rank 1 is the slower replica
        t = bench.max_over_ranks(torch, dist, ws, times[rank], "cpu")
        dist.barrier()
        out[rank] = (t, bench.whole_job_gbs(ws, 36_000_000, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == pytest.approx(0.0075) and res[1][0] == pytest.approx(0.0075)
    assert res[0][1] == pytest.approx(2 * 36_000_000 / 0.0075 / 1e9)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(torch, None, 1, 0.25, "cpu") == 0.25
    assert bench.whole_job_gbs(1, 10 ** 9, 0.5) == pytest.approx(2.0)
