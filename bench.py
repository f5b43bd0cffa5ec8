#!/usr/bin/env python
"""Benchmark: W4A16 decode GEMV throughput (achieved HBM GB/s and fraction of
peak) on the 70B-shaped decode step.

Workload (default): one decode step = 80 layers x {qkv 10240x8192,
o 8192x8192, gate+up fused 57344x8192, down 8192x28672} GEMVs at M = 1,
asymmetric INT4 group-128 weights (N(0, 0.02), drawn on the device, quantized
and packed by the library), bf16 activations N(0,1), f32 accumulation, bf16
outputs.  36.9 GB of packed weights stream from HBM per step, far larger
than L2, so no flush is needed between steps.  The step is captured once as a
CUDA graph of 320 library launches and replayed.

Prints ONE JSON line (rank 0).  Other measurements ride along in "rows":
per-M sweep on the 70B MLP shapes, the quantizer's HBM throughput, and the
large-M GEMM when available.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--M 1] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SIGMA = 0.02
LAYER_SHAPES = [("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192),
                ("down", 8192, 28672)]
METRIC = "W4A16 GEMV achieved HBM GB/s & fraction of peak at M=1..16; us/call"


def algo_bytes(M: int, N: int, K: int, xb: int = 2, yb: int = 2) -> int:
    """Bytes a GEMV must move at minimum: 4-bit codes, one f32 scale and one
    u8 zero per 128 weights, the activations and the outputs."""
    return N * K // 2 + 5 * (N * K // 128) + M * K * xb + M * N * yb


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def profile_traffic(name: str, source_files: list) -> float | None:
    """Per-launch DRAM bytes from a committed ncu summary, or None when the
    kernel source changed since the capture (or no capture exists)."""
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or not h:
        return None
    if h.group(1) != sources_hash(source_files):
        return None
    return float(m.group(1))


def sources_hash(files: list) -> str:
    d = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            d.update(fh.read())
    return d.hexdigest()[:16]


GEMV_SOURCES = ["weight_only_int4_group_gb300/csrc/gemv.cu",
                "weight_only_int4_group_gb300/csrc/common.cuh"]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        self.out.flush()
        rows = []
        with open(self.out.name) as f:
            for line in f:
                p = [s.strip() for s in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.out.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ workload
class Decode70B:
    def __init__(self, q4, torch, M: int, layers: int, seed: int = 1000):
        import synth
        self.q4, self.torch, self.M, self.L = q4, torch, M, layers
        dev = torch.device("cuda")
        self.qw = []  # [layer][matrix] -> QWeight
        wmax = max(N * K for _, N, K in LAYER_SHAPES)
        scratch = torch.empty(wmax, dtype=torch.float32, device=dev)
        for l in range(layers):
            mats = []
            for i, (_, N, K) in enumerate(LAYER_SHAPES):
                w = scratch[:N * K].view(N, K)
                synth.dev_normal_f32(w.data_ptr(), N * K, seed + 4 * l + i, 0, SIGMA)
                packed, scale, zero = q4.quantize(w)
                mats.append(q4.QWeight(q4.repack(packed, scale, zero, N, K), N, K))
                del packed, scale, zero
            self.qw.append(mats)
        del scratch
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        # activations and outputs, one contiguous buffer each (one copy per step e2e)
        self.x_off, self.y_off = [], []
        xo = yo = 0
        for l in range(layers):
            xr, yr = [], []
            for _, N, K in LAYER_SHAPES:
                xr.append(xo)
                yr.append(yo)
                xo += M * K
                yo += M * N
            self.x_off.append(xr)
            self.y_off.append(yr)
        self.x_elems, self.y_elems = xo, yo
        self.x = torch.empty(xo, dtype=torch.int16, device=dev)
        synth.dev_normal_bf16(self.x.data_ptr(), xo, seed + 7777, 0, 1.0)
        self.x = self.x.view(torch.bfloat16)
        self.y = torch.empty(yo, dtype=torch.bfloat16, device=dev)
        # one workspace for every call: each completed call leaves it zero
        wsb = max(q4.gemv_workspace_bytes(M, N, K) for _, N, K in LAYER_SHAPES)
        self.ws = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
        self.bytes_per_step = layers * sum(algo_bytes(M, N, K) for _, N, K in LAYER_SHAPES)
        self.weights_bytes = layers * sum(q4.weight_bytes(N, K) for _, N, K in LAYER_SHAPES)
        self.launches_per_step = layers * len(LAYER_SHAPES)

    def views(self):
        """Per-call (x, y) views into the step's activation and output buffers,
        made once (a caller holds its tensors across steps)."""
        if not hasattr(self, "_views"):
            self._views = [[(self.x[self.x_off[l][i]:self.x_off[l][i] + self.M * K].view(self.M, K),
                             self.y[self.y_off[l][i]:self.y_off[l][i] + self.M * N].view(self.M, N))
                            for i, (_, N, K) in enumerate(LAYER_SHAPES)] for l in range(self.L)]
        return self._views

    def gemv(self, l: int, i: int, path=0):
        x, y = self.views()[l][i]
        self.q4.gemv(x, self.qw[l][i], out=y, ws=self.ws, path=path)

    def step(self, path=0):
        for l in range(self.L):
            for i in range(len(LAYER_SHAPES)):
                self.gemv(l, i, path)


def graph_of(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # eager warm-up (kernel attributes, plans)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, reps: int, warmup: int = 2) -> float:
    """Average seconds per replay, CUDA events on the replaying stream."""
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        g.replay()
    b.record(st)
    b.synchronize()
    return a.elapsed_time(b) / 1e3 / reps


# ------------------------------------------------------------------ CPU oracle
def cpu_sample(M: int, seed: int = 1000, rows_frac: int = 1):
    """Layer 0 of the workload regenerated on the host and quantized by the
    oracle (host threads).  Returns a list of (x, packed, scale, zero, N, K)."""
    import numpy as np

    import oracle
    import synth
    o = oracle.load()
    threads = os.cpu_count() or 1
    out = []
    for i, (_, N, K) in enumerate(LAYER_SHAPES):
        n = N // rows_frac
        W = np.empty((n, K), np.float32)
        bounds = np.linspace(0, n, threads + 1).astype(int)

        def gen(a, b):
            W[a:b] = synth.normal_rows(seed + i, K, a, b, SIGMA)

        ts = [threading.Thread(target=gen, args=(int(bounds[j]), int(bounds[j + 1])))
              for j in range(threads)]
        [t.start() for t in ts]
        [t.join() for t in ts]
        packed = np.empty((n, K // 2), np.uint8)
        scale = np.empty((n, K // 128), np.float32)
        zero = np.empty((n, K // 128), np.uint8)

        def quant(a, b):
            p, s, z = o.quantize(W[a:b])
            packed[a:b], scale[a:b], zero[a:b] = p, s, z

        ts = [threading.Thread(target=quant, args=(int(bounds[j]), int(bounds[j + 1])))
              for j in range(threads) if bounds[j + 1] > bounds[j]]
        [t.start() for t in ts]
        [t.join() for t in ts]
        del W
        x = synth.bf16_bits_to_f32(synth.normal_bf16(seed + 7777 + i, 0, M * K)).reshape(M, K)
        out.append((x, packed, scale, zero, n, K))
    return out, threads


def cpu_pass(sample, threads: int) -> tuple[float, int]:
    import oracle
    o = oracle.load()
    t0 = time.perf_counter()
    nbytes = 0
    for (x, p, s, z, n, K) in sample:
        o.dot_factored(x, p, s, z, n, K, threads=threads)
        nbytes += algo_bytes(x.shape[0], n, K, xb=2, yb=2)
    return time.perf_counter() - t0, nbytes


# ------------------------------------------------------------------ main
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(torch, dist, ws: int, v: float, device) -> float:
    """The largest of every rank's `v` (the slowest replica's time): one
    all-reduce; no collective at all for a single process."""
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(ws: int, bytes_per_replica: int, t_slowest: float) -> float:
    """Aggregate GB/s of `ws` independent replicas, each moving
    `bytes_per_replica` per step, timed by the slowest one."""
    return ws * bytes_per_replica / t_slowest / 1e9


def reference_arm(args, ws, rank):
    """The oracle, as it stands, on the host cores: each step is one pass of
    the page's factored dot over layer 0 of the workload (all four
    matrices), regenerated and quantized on the host."""
    if rank != 0:
        return 0
    sample, threads = cpu_sample(args.M)
    for _ in range(args.warmup):
        cpu_pass(sample, threads)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        t, b = cpu_pass(sample, threads)
        tot_t += t
        tot_b += b
    gbs = tot_b / tot_t / 1e9
    desc = (f"layer 0 of the 70B-shaped decode step (qkv, o, gate+up, down; "
            f"{sum(p.shape[0] * p.shape[1] * 2 for (_, p, _, _, _, _) in sample) / 1e6:.0f} M "
            f"weights), M={args.M}, f32 factored dot of the page, {threads} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"llama70b-shaped decode step, M={args.M}", "M": args.M,
                       "layers_sampled": 1},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--layers", type=int, default=80)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 FMA, 2 MMA")
    ap.add_argument("--no-rows", action="store_true", help="skip the extra measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--case", default=None,
                    help="NxK: time one GEMV shape alone (small-case mode for profilers)")
    ap.add_argument("--reps", type=int, default=3, help="launches in --case mode")
    ap.add_argument("--gemm-case", default=None, help="MxNxK: time one q4_gemm shape alone")
    ap.add_argument("--compact", action="store_true", help="--gemm-case on compact tiles")
    ap.add_argument("--quantize-case", default=None, help="NxK: time q4_quantize on one shape")
    args = ap.parse_args()
    if args.case:
        return single_case(args)
    if args.quantize_case:
        return quantize_case(args)
    if args.gemm_case:
        return gemm_case(args)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        return reference_arm(args, ws, rank)

    import torch
    import torch.distributed as dist

    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import weight_only_int4_group_gb300 as q4

    pk = peaks()
    work = Decode70B(q4, torch, args.M, args.layers)
    g = graph_of(torch, lambda: work.step(args.path))

    # ---- timed region: K replays of the decode-step graph
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    st = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        torch.cuda.synchronize()
        ev0.record(st)
        for _ in range(args.steps):
            g.replay()
        ev1.record(st)
        ev1.synchronize()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_step = max_over_ranks(torch, dist, ws, ev0.elapsed_time(ev1) / 1e3 / args.steps, "cuda")
    assert q4.check() == q4.OK, "device error during the timed region"
    clocks = clk.summary()

    value = whole_job_gbs(ws, work.bytes_per_step, t_step)
    achieved = work.bytes_per_step / t_step / 1e9
    traffic = profile_traffic("gemv_decode70b_M1.md", GEMV_SOURCES) if args.M == 1 else None

    # ---- e2e: public API calls, host buffers, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        hx = torch.empty(work.x_elems, dtype=torch.bfloat16, pin_memory=True)
        hx.copy_(work.x.cpu())
        hy = torch.empty(work.y_elems, dtype=torch.bfloat16, pin_memory=True)
        reps = max(3, min(args.steps // 10, 20))
        for _ in range(2):
            work.x.copy_(hx, non_blocking=True)
            work.step(args.path)
            hy.copy_(work.y, non_blocking=True)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            work.x.copy_(hx, non_blocking=True)
            work.step(args.path)
            hy.copy_(work.y, non_blocking=True)
        b.record(st)
        b.synchronize()
        t_e2e = max_over_ranks(torch, dist, ws, a.elapsed_time(b) / 1e3 / reps, "cuda")
        e2e = {"value": round(whole_job_gbs(ws, work.bytes_per_step, t_e2e), 2), "unit": "GB/s",
               "h2d_bytes_per_step": work.x_elems * 2, "d2h_bytes_per_step": work.y_elems * 2,
               "ms_per_step": round(t_e2e * 1e3, 4), "api": "q4_gemv eager, 320 calls"}

    # ---- extra measurements (rank 0 of a single-GPU run only)
    rows = {}
    if not args.no_rows and rank == 0:
        rows = extra_rows(q4, torch, work, pk)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu:
        sample, threads = cpu_sample(args.M)
        tot_t, tot_b, passes = 0.0, 0, 0
        while tot_t < 2.0 and passes < 50:
            t, b = cpu_pass(sample, threads)
            tot_t, tot_b, passes = tot_t + t, tot_b + b, passes + 1
        cpu = {"value": round(tot_b / tot_t / 1e9, 3), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"layer 0 of the step (4 matrices, 855.6 M weights, host-generated "
                         f"and oracle-quantized), M={args.M}, {passes} passes of the page's f32 "
                         f"factored dot over {threads} threads, {tot_t:.1f} s wall"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"llama70b-shaped decode step: {args.layers} layers x "
                                   f"(qkv 10240x8192, o 8192x8192, gate+up 57344x8192, "
                                   f"down 8192x28672), M={args.M}",
                       "M": args.M, "weights": "int4 asym group-128, f32 scale, u8 zero",
                       "activations": "bf16", "outputs": "bf16", "accumulate": "f32",
                       "arithmetic": "int4 codes x bf16 activations on the tensor cores "
                                     "(mma.sync m16n8k16, bf16 operands), f32 accumulation",
                       "weight_bytes_per_step": work.weights_bytes,
                       "algorithmic_bytes_per_step": work.bytes_per_step,
                       "us_per_token": round(t_step * 1e6, 2),
                       "l2": "inputs (36.9 GB of weights) far larger than L2; no flush",
                       "timing": "CUDA graph of the step, CUDA events on the replay stream",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": traffic, "peak_source": pk["source"],
                         "kernel": "k_gemv (all 320 launches of the step)"},
            "gpu_launches": work.launches_per_step * args.steps,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


def extra_rows(q4, torch, work, pk) -> dict:
    """Per-M sweep on the 70B MLP shapes (80 distinct weight copies, so no L2
    reuse), the quantizer, and the large-M GEMM."""
    rows = {}
    sweep = {}
    L = work.L
    dev = torch.device("cuda")
    for (name, N, K, mi) in (("up 28672x8192", 28672, 8192, 2), ("down 8192x28672", 8192, 28672, 3)):
        # 28672x8192: the first 28672 rows of each fused gate+up weight (row tiles are outermost)
        qws = []
        for l in range(L):
            base = work.qw[l][mi]
            if base.N != N:
                nb = q4.weight_bytes(N, K)
                qws.append(q4.QWeight(base.data[:nb], N, K))
            else:
                qws.append(base)
        res = {}
        for M in (1, 2, 4, 8, 16):
            x = torch.empty(M * K, dtype=torch.int16, device=dev)
            import synth
            synth.dev_normal_bf16(x.data_ptr(), M * K, 4242 + M, 0, 1.0)
            x = x.view(torch.bfloat16).view(M, K)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            wsb = q4.gemv_workspace_bytes(M, N, K)
            wsp = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)

            def run():
                for l in range(L):
                    q4.gemv(x, qws[l], out=y, ws=wsp)
            g = graph_of(torch, run)
            t = time_graph(torch, g, reps=5) / L
            b = algo_bytes(M, N, K)
            res[f"M={M}"] = {"us_per_call": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                             "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4),
                             "weight+scale GB/s": round((N * K // 2 + 5 * N * K // 128) / t / 1e9, 1),
                             "TFLOP/s": round(2 * M * N * K / t / 1e12, 3)}
            del g
        # M = 32: the large-M GEMM, and two M = 16 GEMVs for comparison
        M = 32
        x = torch.empty(M * K, dtype=torch.int16, device=dev)
        synth.dev_normal_bf16(x.data_ptr(), M * K, 4242 + M, 0, 1.0)
        x = x.view(torch.bfloat16).view(M, K)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsp = torch.zeros(max(q4.gemv_workspace_bytes(16, N, K), 256), dtype=torch.uint8, device=dev)
        wsg = torch.zeros(max(q4.gemm_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device=dev)

        def run_gemm():
            for l in range(L):
                q4.gemm(x, qws[l], out=y, ws=wsg)

        def run_two():
            for l in range(L):
                q4.gemv(x[:16], qws[l], out=y[:16], ws=wsp)
                q4.gemv(x[16:], qws[l], out=y[16:], ws=wsp)
        b = algo_bytes(M, N, K)
        for rname, fn in (("M=32 q4_gemm", run_gemm), ("M=32 as 2 x M=16 q4_gemv", run_two)):
            g = graph_of(torch, fn)
            t = time_graph(torch, g, reps=5) / L
            res[rname] = {"us_per_call": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                          "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4),
                          "TFLOP/s": round(2 * M * N * K / t / 1e12, 3)}
            del g
        # M = 1 through each kernel explicitly (AUTO picks the tensor-core one)
        x = torch.empty(K, dtype=torch.int16, device=dev)
        synth.dev_normal_bf16(x.data_ptr(), K, 4242, 0, 1.0)
        x = x.view(torch.bfloat16).view(1, K)
        y = torch.empty((1, N), dtype=torch.bfloat16, device=dev)
        wsp = torch.zeros(max(q4.gemv_workspace_bytes(1, N, K), 256), dtype=torch.uint8, device=dev)
        for pname, pid in (("M=1 cuda-core FMA", q4.PATH_FMA), ("M=1 tensor-core MMA", q4.PATH_MMA)):
            def runp():
                for l in range(L):
                    q4.gemv(x, qws[l], out=y, ws=wsp, path=pid)
            g = graph_of(torch, runp)
            t = time_graph(torch, g, reps=5) / L
            b = algo_bytes(1, N, K)
            res[pname] = {"us_per_call": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                          "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4)}
            del g
        sweep[name] = res
    rows["mlp_sweep"] = sweep

    # compact tiles (binary16 scales, 4-bit zeros) on 28672x8192: as many
    # distinct copies as the sweep above used (far beyond L2, the same graph
    # length); bytes counted as the compact tiles actually read, and the time
    # per call set against the same M above
    import synth
    N, K, C = 28672, 8192, L
    wf = torch.empty((N, K), dtype=torch.float32, device=dev)
    synth.dev_normal_f32(wf.data_ptr(), N * K, 777, 0, SIGMA)
    packed, scale, zero = q4.quantize(wf)
    del wf
    cqws = [q4.QWeight(q4.repack_compact(packed, scale, zero, N, K), N, K, compact=True)
            for _ in range(C)]
    del packed, scale, zero
    cres = {}
    for M in (1, 8, 16):
        x = torch.empty(M * K, dtype=torch.int16, device=dev)
        synth.dev_normal_bf16(x.data_ptr(), M * K, 4242 + M, 0, 1.0)
        x = x.view(torch.bfloat16).view(M, K)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        wsp = torch.zeros(max(q4.gemv_workspace_bytes(M, N, K), 256), dtype=torch.uint8, device=dev)

        def runc():
            for c in range(C):
                q4.gemv(x, cqws[c], out=y, ws=wsp)
        g = graph_of(torch, runc)
        t = time_graph(torch, g, reps=10) / C
        b = q4.weight_bytes_compact(N, K) + M * K * 2 + M * N * 2
        std = sweep["up 28672x8192"][f"M={M}"]["us_per_call"]
        cres[f"M={M}"] = {"us_per_call": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                          "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4),
                          "speedup_vs_1104B_tiles": round(std / (t * 1e6), 4)}
        del g
    rows["compact_28672x8192"] = cres
    del cqws
    torch.cuda.empty_cache()

    # the decode step at M = 8 on the same weights (80 layers, one graph)
    M = 8
    import synth
    xs, ys = [], []
    for _, N, K in LAYER_SHAPES:
        xb = torch.empty(M * K, dtype=torch.int16, device=dev)
        synth.dev_normal_bf16(xb.data_ptr(), M * K, 808 + K, 0, 1.0)
        xs.append(xb.view(torch.bfloat16).view(M, K))
        ys.append(torch.empty((M, N), dtype=torch.bfloat16, device=dev))
    ws8 = torch.zeros(max(256, max(q4.gemv_workspace_bytes(M, N, K) for _, N, K in LAYER_SHAPES)),
                      dtype=torch.uint8, device=dev)

    def step8():
        for l in range(L):
            for i, (_, N, K) in enumerate(LAYER_SHAPES):
                q4.gemv(xs[i], work.qw[l][i], out=ys[i], ws=ws8)
    g = graph_of(torch, step8)
    t = time_graph(torch, g, reps=3)
    b = L * sum(algo_bytes(M, N, K) for _, N, K in LAYER_SHAPES)
    rows["decode_step_M8"] = {"layers": L, "ms_per_step": round(t * 1e3, 3),
                              "GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4)}
    del g, xs, ys, ws8

    # Llama-7B-shaped layer, M = 1 (qkv 12288x4096, o 4096x4096, gate and up
    # 11008x4096 each, down 4096x11008; 0.1% of input channels x20): gate and
    # up read the same activations and run as one 22016x4096 GEMV (their
    # tiled buffers concatenated along the rows, as for the 70B step); 8
    # distinct layers per graph (0.87 GB, beyond L2), time per layer
    mats7 = [("qkv", 12288, 4096), ("o", 4096, 4096), ("gate", 11008, 4096), ("up", 11008, 4096),
             ("down", 4096, 11008)]
    shapes7 = [("qkv", 12288, 4096), ("o", 4096, 4096), ("gate_up", 22016, 4096),
               ("down", 4096, 11008)]
    L7 = 8
    q7 = []
    for l in range(L7):
        mats = []
        for i, (_, N, K) in enumerate(mats7):
            w = torch.empty((N, K), dtype=torch.float32, device=dev)
            cols = torch.from_numpy(synth.outlier_columns(70 + i, K).astype("int64")).to(dev)
            synth.dev_normal_f32(w.data_ptr(), N * K, 7000 + 10 * l + i, 0, SIGMA)
            w[:, cols] *= 20.0
            mats.append(q4.QWeight.from_float(w))
            del w
        gate, up = mats[2], mats[3]
        mats[2:4] = [q4.QWeight(torch.cat([gate.data, up.data]), gate.N + up.N, gate.K)]
        q7.append(mats)
    x7 = {}
    for _, N, K in shapes7:
        if K not in x7:
            xb = torch.empty(K, dtype=torch.int16, device=dev)
            synth.dev_normal_bf16(xb.data_ptr(), K, 707 + K, 0, 1.0)
            x7[K] = xb.view(torch.bfloat16).view(1, K)
    y7 = [torch.empty((1, N), dtype=torch.bfloat16, device=dev) for _, N, _ in shapes7]
    ws7 = torch.zeros(max(256, max(q4.gemv_workspace_bytes(1, N, K) for _, N, K in shapes7)),
                      dtype=torch.uint8, device=dev)

    def layer7():
        for l in range(L7):
            for i, (_, N, K) in enumerate(shapes7):
                q4.gemv(x7[K], q7[l][i], out=y7[i], ws=ws7)
    g = graph_of(torch, layer7)
    t = time_graph(torch, g, reps=10) / L7
    b = sum(algo_bytes(1, N, K) for _, N, K in shapes7)
    rows["llama7b_layer_M1"] = {"us_per_layer": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                                "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4),
                                "launches_per_layer": len(shapes7)}
    del g, q7, x7, y7, ws7

    # single GEMV, 4096 x 4096, the page's xorshift matrix, f32 x and y, M = 1:
    # one copy repeated (L2-resident) and 48 copies rotated (0.44 GB, beyond L2)
    W1, xv = synth.xorshift_matrix(4096, 4096)
    w1 = torch.from_numpy(W1).to(dev)
    q1 = q4.QWeight.from_float(w1)
    del w1
    x1 = torch.from_numpy(xv.reshape(1, -1)).to(dev)
    y1 = torch.empty((1, 4096), dtype=torch.float32, device=dev)
    copies = [q1] + [q4.QWeight(q1.data.clone(), 4096, 4096) for _ in range(47)]
    ws1 = torch.zeros(max(q4.gemv_workspace_bytes(1, 4096, 4096), 256), dtype=torch.uint8, device=dev)
    b = algo_bytes(1, 4096, 4096, xb=4, yb=4)
    single = {}
    for rname, seq in (("L2-resident (one copy)", [q1] * 48), ("rotated (48 copies)", copies)):
        def run1():
            for qq in seq:
                q4.gemv(x1, qq, out=y1, ws=ws1)
        g = graph_of(torch, run1)
        t = time_graph(torch, g, reps=10) / len(seq)
        single[rname] = {"us_per_call": round(t * 1e6, 2), "GB/s": round(b / t / 1e9, 1),
                         "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4)}
        del g
    rows["single_4096x4096_f32"] = single
    del copies, q1, x1, y1, ws1

    # large-M GEMM (prefill): 4096 tokens x 8192 x 28672, tcgen05 tensor cores
    Mg, Ng, Kg = 4096, 28672, 8192
    qg = work.qw[0][2]  # first 28672 rows of a fused gate+up weight
    qg = q4.QWeight(qg.data[:q4.weight_bytes(Ng, Kg)], Ng, Kg)
    xg = torch.empty(Mg * Kg, dtype=torch.int16, device=dev)
    synth.dev_normal_bf16(xg.data_ptr(), Mg * Kg, 777, 0, 1.0)
    xg = xg.view(torch.bfloat16).view(Mg, Kg)
    yg = torch.empty((Mg, Ng), dtype=torch.bfloat16, device=dev)

    wsg = torch.zeros(max(256, q4.gemm_workspace_bytes(Mg, Ng, Kg)), dtype=torch.uint8, device=dev)
    flops = 2.0 * Mg * Ng * Kg
    for rname, qq in (("gemm_prefill", qg), ("gemm_prefill_compact", None)):
        if qq is None:  # the same weights in compact tiles (binary16 scales, 4-bit zeros)
            wf = torch.empty((Ng, Kg), dtype=torch.float32, device=dev)
            synth.dev_normal_f32(wf.data_ptr(), Ng * Kg, 1000 + 2, 0, SIGMA)
            qq = q4.QWeight.from_float(wf, compact=True)
            del wf

        def grun(qq=qq):
            q4.gemm(xg, qq, out=yg, ws=wsg)
        g = graph_of(torch, grun)
        t = time_graph(torch, g, reps=10)
        rows[rname] = {"shape": f"M={Mg} N={Ng} K={Kg} bf16",
                       "operands": "binary16 weights (one rounding) and activations (exact) behind "
                                   "power-of-two row/token scalings, f32 accumulation; prep, GEMM "
                                   "and scratch-clear passes all timed",
                       "ms": round(t * 1e3, 3),
                       "TFLOP/s": round(flops / t / 1e12, 1),
                       "frac_of_bf16_peak": round(flops / t / 1e12 / pk["bf16_tflops"], 4),
                       "peak": pk["bf16_tflops"], "peak_kind": "burst, of measured"}
        del g
    del xg, yg, wsg
    torch.cuda.empty_cache()

    # quantizers (asymmetric, symmetric): HBM-bound, 4 B read + 0.539 B
    # written per weight
    N, K = 57344, 8192
    import synth
    w = torch.empty((N, K), dtype=torch.float32, device=dev)
    synth.dev_normal_f32(w.data_ptr(), N * K, 99, 0, SIGMA)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scale = torch.empty((N, K // 128), dtype=torch.float32, device=dev)
    zero = torch.empty((N, K // 128), dtype=torch.uint8, device=dev)
    lib = q4.lib()

    b = 4 * N * K + N * K // 2 + 5 * N * K // 128
    for key, fn in (("quantize", lib.q4_quantize), ("quantize_sym", lib.q4_quantize_sym)):
        def qrun(fn=fn):
            fn(w.data_ptr(), N, K, packed.data_ptr(), scale.data_ptr(), zero.data_ptr(),
               torch.cuda.current_stream().cuda_stream)
        g = graph_of(torch, qrun)
        t = time_graph(torch, g, reps=10)
        rows[key] = {"shape": f"{N}x{K} f32", "ms": round(t * 1e3, 3),
                     "GB/s": round(b / t / 1e9, 1), "frac": round(b / t / 1e9 / pk["hbm_gbs"], 4)}
        del g
    del w, packed, scale, zero
    torch.cuda.empty_cache()
    return rows


def single_case(args) -> int:
    """One GEMV shape, `reps` launches on a few distinct weight copies (more
    than L2 in total), printed as a plain JSON line.  Used to give profilers
    a small, self-contained command."""
    import torch

    import synth
    import weight_only_int4_group_gb300 as q4
    N, K = (int(v) for v in args.case.lower().split("x"))
    M = args.M
    dev = torch.device("cuda")
    copies = max(1, -(-3 * 129_000_000 // q4.weight_bytes(N, K)))  # >= 3x L2 in total
    w = torch.empty((N, K), dtype=torch.float32, device=dev)
    qws = []
    for c in range(copies):
        synth.dev_normal_f32(w.data_ptr(), N * K, 500 + c, 0, SIGMA)
        qws.append(q4.QWeight.from_float(w))
    del w
    x = torch.empty(M * K, dtype=torch.int16, device=dev)
    synth.dev_normal_bf16(x.data_ptr(), M * K, 501, 0, 1.0)
    x = x.view(torch.bfloat16).view(M, K)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = q4.workspace(M, N, K)
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(copies):  # warm-up: one launch per copy
        q4.gemv(x, qws[i], out=y, ws=ws, path=args.path)
    torch.cuda.synchronize()
    a.record(st)
    for i in range(args.reps):
        q4.gemv(x, qws[i % copies], out=y, ws=ws, path=args.path)
    b.record(st)
    b.synchronize()
    assert q4.check() == q4.OK
    t = a.elapsed_time(b) / 1e3 / args.reps
    nb = algo_bytes(M, N, K)
    print(json.dumps({"case": f"{N}x{K}", "M": M, "path": args.path, "copies": copies,
                      "launches": copies + args.reps, "us_per_call": round(t * 1e6, 2),
                      "GB/s": round(nb / t / 1e9, 1)}), flush=True)
    return 0


def quantize_case(args) -> int:
    """q4_quantize on one N x K f32 matrix (device-generated), `reps` launches
    after one warm-up, printed as a plain JSON line."""
    import torch

    import synth
    import weight_only_int4_group_gb300 as q4
    N, K = (int(v) for v in args.quantize_case.lower().split("x"))
    dev = torch.device("cuda")
    w = torch.empty((N, K), dtype=torch.float32, device=dev)
    synth.dev_normal_f32(w.data_ptr(), N * K, 99, 0, SIGMA)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    scale = torch.empty((N, K // 128), dtype=torch.float32, device=dev)
    zero = torch.empty((N, K // 128), dtype=torch.uint8, device=dev)
    lib = q4.lib()

    def run():
        rc = lib.q4_quantize(w.data_ptr(), N, K, packed.data_ptr(), scale.data_ptr(),
                             zero.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == q4.OK, rc
    run()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        run()
    b.record()
    b.synchronize()
    t = a.elapsed_time(b) / 1e3 / args.reps
    nb = 4 * N * K + N * K // 2 + 5 * N * K // 128
    print(json.dumps({"quantize_case": f"{N}x{K}", "us": round(t * 1e6, 2),
                      "GB/s": round(nb / t / 1e9, 1)}), flush=True)
    return 0


def gemm_case(args) -> int:
    """One q4_gemm shape (bf16), `reps` launches after one warm-up."""
    import torch

    import synth
    import weight_only_int4_group_gb300 as q4
    M, N, K = (int(v) for v in args.gemm_case.lower().split("x"))
    dev = torch.device("cuda")
    w = torch.empty((N, K), dtype=torch.float32, device=dev)
    synth.dev_normal_f32(w.data_ptr(), N * K, 600, 0, SIGMA)
    qw = q4.QWeight.from_float(w, compact=args.compact)
    del w
    x = torch.empty(M * K, dtype=torch.int16, device=dev)
    synth.dev_normal_bf16(x.data_ptr(), M * K, 601, 0, 1.0)
    x = x.view(torch.bfloat16).view(M, K)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = q4.gemm_workspace(M, N, K)
    q4.gemm(x, qw, out=y, ws=ws)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.reps):
        q4.gemm(x, qw, out=y, ws=ws)
    b.record()
    b.synchronize()
    assert q4.check() == q4.OK
    t = a.elapsed_time(b) / 1e3 / args.reps
    print(json.dumps({"gemm_case": f"{M}x{N}x{K}", "ms": round(t * 1e3, 3),
                      "TFLOP/s": round(2.0 * M * N * K / t / 1e12, 1),
                      "GB/s": round(algo_bytes(M, N, K) / t / 1e9, 1)}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
