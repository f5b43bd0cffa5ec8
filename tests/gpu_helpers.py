"""Helpers shared by the GPU parity tests: moving seeded inputs to the device,
running the oracle, and the comparison rule.

Comparison rule for GEMV/GEMM outputs (per element):
    |y_gpu - y_oracle| <= 1e-3 * sum_k |w_hat * x| + 1e-5
with sum_k |w_hat * x| computed in double by the oracle.  For bf16/f16
outputs both sides are rounded to the output type first (round to nearest
even from f32), and one unit in the last place of the rounded oracle value is
added to the allowance: two values on either side of a rounding boundary may
round one ulp apart even when they agree to far better than the tolerance.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

RTOL = 1e-3
ATOL = 1e-5


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def dev_bf16_bits(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def x_for(dtype, M: int, K: int, seed: int = 11):
    """Activations ~ N(0,1) in `dtype`: (device tensor, exact f32 copy on host)."""
    if dtype == torch.bfloat16:
        bits = synth.normal_bf16(seed, 0, M * K).reshape(M, K)
        return dev_bf16_bits(bits), synth.bf16_bits_to_f32(bits)
    f = synth.normal(seed, 0, M * K).reshape(M, K)
    if dtype == torch.float16:
        h = f.astype(np.float16)
        return torch.from_numpy(h).cuda(), h.astype(np.float32)
    return dev_f32(f), f


def round_to(y: np.ndarray, dtype) -> np.ndarray:
    """Round f32/f64 values to `dtype` (RNE from f32) and back to f64."""
    y32 = np.asarray(y, np.float32)
    if dtype == torch.float32:
        return y32.astype(np.float64)
    return torch.from_numpy(y32).to(dtype).to(torch.float64).numpy()


def ulp_of(v: np.ndarray, dtype) -> np.ndarray:
    if dtype == torch.float32:
        return np.zeros_like(v)
    mant = 8 if dtype == torch.bfloat16 else 11
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    if dtype == torch.float16:
        e = np.maximum(e, -14)
    return np.where(a > 0, 2.0 ** (e - (mant - 1)), 0.0)


def compare(y_gpu: torch.Tensor, y_ref: np.ndarray, absdot: np.ndarray, where: str = "") -> dict:
    dt = y_gpu.dtype
    g = y_gpu.float().cpu().numpy().astype(np.float64)
    r = round_to(y_ref, dt)
    tol = RTOL * absdot + ATOL
    allow = tol + ulp_of(r, dt)
    err = np.abs(g - r)
    bad = err > allow
    used_ulp = int(((err > tol) & ~bad).sum())
    assert not bad.any(), (
        f"{where}: {int(bad.sum())} of {bad.size} outside tolerance; worst err/allow "
        f"{float((err / allow).max()):.3g} at {np.unravel_index(np.argmax(err / allow), err.shape)}")
    return {"max_err_over_tol": float((err / tol).max()), "ulp_allowance_used": used_ulp}


def oracle_product(W: np.ndarray, Xf: np.ndarray, threads: int = 8):
    o = oracle.load()
    N, K = W.shape
    p, s, z = o.quantize(W)
    y, a = o.dot_naive(Xf, p, s, z, N, K, threads=threads)
    return (p, s, z), y, a
