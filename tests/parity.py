"""Helpers for GPU-vs-oracle parity tests.

Tolerances (per output element, against the fp64 oracle):
    fp32 I/O:  |y - y_ref| <= 1e-4 * (1 + |y_ref|)
    bf16 I/O:  |y - y_ref| <= 2e-2 * (1 + |y_ref|)   (fp32 state, bf16 rounding of y)
last_state (always fp32) meets the bound of the I/O type it was computed from.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import selective_state_space_116_b300 as ssm

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def nthreads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def to_cuda(inp: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def gpu_scan(inp: dict, chunk: int = 0, return_last_state: bool = True, **opts):
    g = to_cuda(inp)
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                            delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                            return_last_state=return_last_state, chunk=chunk, check=True,
                            **opts)
    torch.cuda.synchronize()
    return y, h


def oracle_scan(inp: dict, channels=None):
    return oracle.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                           z=inp["z"], delta_bias=inp["delta_bias"],
                           delta_softplus=inp["delta_softplus"], channels=channels,
                           nthreads=nthreads())


def as64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, io_dtype, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    tol = TOL[io_dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = tol * (1.0 + np.abs(ref))
    ratio = err / bound
    worst = np.unravel_index(np.argmax(ratio), ratio.shape) if ratio.size else None
    assert not (ratio > 1.0).any(), (
        f"{what}: {(ratio > 1).sum()} of {ratio.size} outside tol {tol}; worst at {worst}: "
        f"got {got[worst]:.6g} ref {ref[worst]:.6g}")
    return float(ratio.max()) if ratio.size else 0.0


def sample_channels(batch: int, dim: int, k: int = 64, seed: int = 0):
    """k flat channel ids, always including the first and last channel of every batch row."""
    rng = np.random.default_rng(seed)
    must = sorted({b * dim for b in range(batch)} | {b * dim + dim - 1 for b in range(batch)})
    rest = rng.choice(batch * dim, size=max(0, k - len(must)), replace=False)
    return np.array(sorted(set(must) | set(int(c) for c in rest)), dtype=np.int64)
