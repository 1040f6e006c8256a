"""Unrolled O(L^2) selective-scan sum -- TEST INFRASTRUCTURE ONLY.

A second, independent statement of the scan for tiny inputs.  It does not
step the recurrence; it writes out its general solution.  Unrolling
h_t = Abar_t h_{t-1} + Bbar_t x_t from h_{-1} = 0 (the recurrence of the
elemedex "Mamba" entry, section "How it works", with Abar_t = exp(Delta_t A)
and Bbar_t x_t = Delta_t B_t x_t) gives

    h_{t,n} = sum_{s<=t} exp(A_n * sum_{r=s+1..t} Delta_r) * Delta_s * B_{s,n} * u_s
    y_t     = (sum_n C_{t,n} h_{t,n} + D u_t) * silu(z_t)

which is evaluated here as a dense (t, s) matrix with numpy.  Softplus and
the sigmoid come from numpy/scipy library routines (``logaddexp``,
``expit``), not from the C oracle's own formulas.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
             zoh=False, h0=None):
    """u, delta, z: (batch, dim, L); B, C: (batch, L, N); A: (dim, N).
    zoh: the exact zero-order-hold input weight expm1(Delta_s A_n) / A_n in
    place of Delta_s (Delta_s where A_n = 0).  h0: (batch, dim, N) initial
    state, carried to token t by exp(A_n * sum_{r<=t} Delta_r).
    Returns (y (batch, dim, L), last_state (batch, dim, N)) in fp64."""
    u = np.asarray(u, np.float64)
    delta = np.asarray(delta, np.float64)
    A = np.asarray(A, np.float64)
    B = np.asarray(B, np.float64)
    C = np.asarray(C, np.float64)
    batch, dim, L = u.shape
    N = A.shape[1]
    v = delta + (0.0 if delta_bias is None else np.asarray(delta_bias, np.float64)[None, :, None])
    dt = np.logaddexp(0.0, v) if delta_softplus else v               # (batch, dim, L)
    S = np.cumsum(dt, axis=-1)                                       # S_t = sum_{r<=t} dt_r
    gap = S[..., :, None] - S[..., None, :]                          # (b, d, t, s): sum_{s<r<=t}
    causal = np.tril(np.ones((L, L), dtype=bool))
    # decay[b,d,t,s,n] = exp(A_n * gap) for s <= t, else 0 (exp(-inf))
    expo = A[None, :, None, None, :] * gap[..., None]
    decay = np.exp(np.where(causal[None, None, :, :, None], expo, -np.inf))
    if zoh:   # weight[b,d,s,n] = expm1(dt_s A_n) / A_n, or dt_s where A_n = 0
        prod = dt[..., None] * A[None, :, None, :]
        safe = np.where(A == 0.0, 1.0, A)[None, :, None, :]
        weight = np.where(A[None, :, None, :] == 0.0, dt[..., None], np.expm1(prod) / safe)
    else:
        weight = np.broadcast_to(dt[..., None], dt.shape + (N,))
    drive = (weight * u[..., None]) * B[:, None, :, :]                # (b, d, s, n)
    h = np.einsum("bdtsn,bdsn->bdtn", decay, drive)                   # (b, d, t, n)
    if h0 is not None:   # the initial state decays by exp(A_n S_t)
        h = h + np.exp(A[None, :, None, :] * S[..., None]) * np.asarray(h0, np.float64)[:, :, None, :]
    y = np.einsum("btn,bdtn->bdt", C, h)
    if D is not None:
        y = y + np.asarray(D, np.float64)[None, :, None] * u
    if z is not None:
        z = np.asarray(z, np.float64)
        y = y * (z * expit(z))
    if L == 0:
        return y, (np.zeros((batch, dim, N)) if h0 is None else np.array(h0, np.float64))
    return y, h[:, :, -1, :].copy()
