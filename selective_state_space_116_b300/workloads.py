"""Seeded synthetic inputs for the selective scan.

This module only draws random numbers and lays them out; it holds none of
the scan's arithmetic.  Both the CUDA library's tests/benchmark and the CPU
oracle read the tensors it returns, so the two sides always see identical
inputs.

Recipe (all workloads): numpy ``default_rng(seed)`` (PCG64), values drawn in
fp32 in the order u, delta, A, B, C, D, delta_bias, z, then rounded to the
I/O dtype with round-to-nearest-even.  ``delta`` is the raw pre-activation:
the step size the scan uses is softplus(delta + delta_bias) when
``delta_softplus`` is set.  A, D and delta_bias are always fp32.

Layouts: u, delta, z, y: (batch, dim, L), L contiguous; B, C: (batch, L, N);
A: (dim, N); D, delta_bias: (dim,); state: (batch, dim, N).

Workloads, named after the Mamba layer sizes they imitate:

* ``tiny``  1 x 16 channels, N=4, L=256, fp32; u~N(0,1); delta~N(0,1)-2
  with softplus and no bias; A=-exp(U(0,1.5)); B,C~N(0,1); D~N(0,1); no z.
* ``m130``  Mamba-130M layer: 8 x 1536, N=16, L=2048, bf16 I/O; u,z~N(0,1);
  delta~N(0,1); bias~U(-4,-2) with softplus; A_n=-(n+1); B,C,D~N(0,1).
* ``m2p8``  Mamba-2.8B layer: 4 x 5120, N=16, L=4096, otherwise as m130.
* ``dna``   long DNA-like sequence: 1 x 1024, N=16, L=2^20, fp32 I/O; a
  symbol stream s_t~U{0..3}; u[d,t] = g_d if s_t == d mod 4 else 0 with
  g_d~N(0,1) (one-hot over four symbols times a per-channel gain);
  delta~N(-3,1) with softplus, no bias; A=-exp(U(0,1.5)); B,C,D~N(0,1).
* ``gen``   generation: 128 x 5120, N=16, one token per step, bf16 x/delta/
  z/B/C, fp32 state, bias~U(-4,-2) with softplus, A_n=-(n+1), D~N(0,1).

The selective-copying experiment of "Mamba remembers by forgetting, read
closely" (interactiveml.org) has its own generator, ``selective_copy_inputs``:
a target scalar followed by Gaussian distractors, with a fixed or a
selective step size.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    io: str                      # "f32" or "bf16"
    delta_mean: float = 0.0      # raw delta ~ N(delta_mean, 1)
    bias_range: tuple | None = None   # delta_bias ~ U(lo, hi), or None
    softplus: bool = True
    a_kind: str = "neg_exp_uniform"   # or "neg_index": A_n = -(n+1)
    gate: bool = False           # z ~ N(0,1) present
    skip: bool = True            # D ~ N(0,1) present
    u_kind: str = "normal"       # or "onehot4"
    last_state: bool = True
    steps: int = 0               # generation workloads: number of tokens

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def torch_io(self):
        return torch.bfloat16 if self.io == "bf16" else torch.float32


WORKLOADS = {
    "tiny": Workload("tiny", 1, 16, 4, 256, "f32", delta_mean=-2.0, bias_range=None),
    "m130": Workload("m130", 8, 1536, 16, 2048, "bf16", bias_range=(-4.0, -2.0),
                     a_kind="neg_index", gate=True, last_state=False),
    "m2p8": Workload("m2p8", 4, 5120, 16, 4096, "bf16", bias_range=(-4.0, -2.0),
                     a_kind="neg_index", gate=True),
    "dna": Workload("dna", 1, 1024, 16, 1 << 20, "f32", delta_mean=-3.0, bias_range=None,
                    u_kind="onehot4"),
    "gen": Workload("gen", 128, 5120, 16, 1, "bf16", bias_range=(-4.0, -2.0),
                    a_kind="neg_index", gate=True, steps=1024),
}


def _normal(rng, shape, mean=0.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if mean:
        x += np.float32(mean)
    return x


def _to_io(x: np.ndarray, dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype)


def _params(w: Workload, rng):
    if w.a_kind == "neg_index":
        A = -np.tile(np.arange(1, w.dstate + 1, dtype=np.float32), (w.dim, 1))
    else:
        A = -np.exp(rng.uniform(0.0, 1.5, size=(w.dim, w.dstate)).astype(np.float32))
    return np.ascontiguousarray(A, dtype=np.float32)


def make_scan_inputs(w: Workload, seed: int = 0) -> dict:
    """Host (CPU) tensors for one forward scan of workload ``w``."""
    rng = np.random.default_rng(seed)
    b, d, L, N = w.batch, w.dim, w.seqlen, w.dstate
    io = w.torch_io
    if w.u_kind == "onehot4":
        sym = rng.integers(0, 4, size=L)
        gain = rng.standard_normal(size=d, dtype=np.float32)
        hit = sym[None, :] == (np.arange(d) % 4)[:, None]            # (d, L)
        u = np.where(hit, gain[:, None], np.float32(0.0)).astype(np.float32)[None]
        u = np.broadcast_to(u, (b, d, L)).copy()
    else:
        u = _normal(rng, (b, d, L))
    delta = _normal(rng, (b, d, L), w.delta_mean)
    A = _params(w, rng)
    B = _normal(rng, (b, L, N))
    C = _normal(rng, (b, L, N))
    D = _normal(rng, (d,)) if w.skip else None
    bias = (rng.uniform(*w.bias_range, size=d).astype(np.float32)
            if w.bias_range is not None else None)
    z = _normal(rng, (b, d, L)) if w.gate else None
    return {
        "u": _to_io(u, io), "delta": _to_io(delta, io),
        "A": torch.from_numpy(A), "B": _to_io(B, io), "C": _to_io(C, io),
        "D": None if D is None else torch.from_numpy(D),
        "z": None if z is None else _to_io(z, io),
        "delta_bias": None if bias is None else torch.from_numpy(bias),
        "delta_softplus": w.softplus,
    }


def make_step_inputs(w: Workload, seed: int = 0, steps: int | None = None) -> dict:
    """Host tensors for ``steps`` consecutive single-token updates.

    Per-step inputs are stacked along a leading step axis so that each step's
    slice is contiguous: x, delta, z (steps, batch, dim); B, C (steps, batch, N).
    """
    rng = np.random.default_rng(seed)
    T = w.steps if steps is None else steps
    b, d, N = w.batch, w.dim, w.dstate
    io = w.torch_io
    x = _normal(rng, (T, b, d))
    delta = _normal(rng, (T, b, d), w.delta_mean)
    A = _params(w, rng)
    B = _normal(rng, (T, b, N))
    C = _normal(rng, (T, b, N))
    D = _normal(rng, (d,)) if w.skip else None
    bias = (rng.uniform(*w.bias_range, size=d).astype(np.float32)
            if w.bias_range is not None else None)
    z = _normal(rng, (T, b, d)) if w.gate else None
    return {
        "x": _to_io(x, io), "delta": _to_io(delta, io),
        "A": torch.from_numpy(A), "B": _to_io(B, io), "C": _to_io(C, io),
        "D": None if D is None else torch.from_numpy(D),
        "z": None if z is None else _to_io(z, io),
        "delta_bias": None if bias is None else torch.from_numpy(bias),
        "delta_softplus": w.softplus,
    }


def steps_as_scan(inp: dict) -> dict:
    """The same token stream laid out as one scan: x (T, b, d) -> u (b, d, T),
    B (T, b, N) -> (b, T, N).  Pure re-layout of the drawn values."""
    def tr(t, perm):
        return None if t is None else t.permute(*perm).contiguous()
    return {
        "u": tr(inp["x"], (1, 2, 0)), "delta": tr(inp["delta"], (1, 2, 0)),
        "A": inp["A"], "B": tr(inp["B"], (1, 0, 2)), "C": tr(inp["C"], (1, 0, 2)),
        "D": inp["D"], "z": tr(inp["z"], (1, 2, 0)), "delta_bias": inp["delta_bias"],
        "delta_softplus": inp["delta_softplus"],
    }


# The step sizes of the selective-copying experiment: one fixed step for every
# item, or a large step on the target and a tiny one on the distractors
# ("Mamba remembers by forgetting, read closely", interactiveml.org, the
# selective-copying paragraphs).
COPY_FIXED_DELTA = 0.25
COPY_TARGET_DELTA = 6.0
COPY_NOISE_DELTA = 0.002


def selective_copy_inputs(gap: int, n_seq: int = 400, seed: int = 0, selective: bool = True) -> dict:
    """Host tensors for the selective-copying experiment at one gap.

    Each of the ``n_seq`` independently drawn sequences is one channel: token 0
    is the target x_0 ~ N(0, 1), tokens 1..gap are distractors ~ N(0, 1).  The
    scan is the page's scalar recurrence (N = 1, A = -1, B = C = 1, no skip
    term, no gate, Delta given directly), to be run with the exact zero-order
    hold input term, so that y[0, d, t] is the state after token t and
    y[0, d, gap] is what the memory holds when the target is recalled.
    Delta is 0.25 everywhere (fixed), or 6 on the target and 0.002 on the
    distractors (selective).  The same seed gives the same sequences in both
    settings.  Returns the scan inputs plus ``target`` (n_seq,).
    """
    rng = np.random.default_rng(seed)
    L = gap + 1
    x = _normal(rng, (1, n_seq, L))
    delta = np.full((1, n_seq, L), COPY_NOISE_DELTA if selective else COPY_FIXED_DELTA,
                    dtype=np.float32)
    if selective:
        delta[..., 0] = COPY_TARGET_DELTA
    return {
        "u": torch.from_numpy(x), "delta": torch.from_numpy(delta),
        "A": torch.full((n_seq, 1), -1.0), "B": torch.ones(1, L, 1), "C": torch.ones(1, L, 1),
        "D": None, "z": None, "delta_bias": None, "delta_softplus": False,
        "target": torch.from_numpy(x[0, :, 0].copy()),
    }
