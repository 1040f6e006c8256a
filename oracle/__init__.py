"""Selective-scan oracle (fp64, CPU) -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never loads it, and it shares no code
with the CUDA library: the arithmetic lives in ``ssm_oracle.c`` (plain C,
fp64, sequential per channel) and in ``brute.py`` (an independent O(L^2)
closed-form sum for tiny inputs).

``build()`` compiles ``ssm_oracle.c`` with gcc into ``libssm_oracle.so`` next
to it (``-O2``, no fast-math, so every ``exp``/``log1p`` is the C library's
fp64 routine).  The wrappers below only marshal arrays: they hand the host
buffers (fp32, bf16 bit patterns, or fp64) straight to the C code, which
widens or decodes each element itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ssm_oracle.c")
LIBRARY = os.path.join(_HERE, "libssm_oracle.so")

# element type codes understood by ssm_oracle.c
F32, BF16, F64 = 0, 1, 2

_lib_cache: dict[str, ctypes.CDLL] = {}


def build(source: str = SOURCE, out: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle C source into a shared library (skipped if fresh)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
         "-o", tmp, source, "-lm"],
        check=True,
    )
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) an oracle library; cached per path."""
    if path is None:
        path = build()
    if path not in _lib_cache:
        lib = ctypes.CDLL(path)
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        lib.oracle_scan_fwd.restype = i32
        lib.oracle_scan_fwd.argtypes = [i64, i64, i64, i64, i32, i32,
                                        vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                        vp, i64, dp, dp, dp, i32]
        lib.oracle_state_step.restype = i32
        lib.oracle_state_step.argtypes = [i64, i64, i64, i32, i32,
                                          dp, vp, vp, vp, vp, vp, vp, vp, vp, i32, dp]
        lib.oracle_conv_silu.restype = i32
        lib.oracle_conv_silu.argtypes = [i64, i64, i64, i64, i32, i32, vp, vp, vp, vp, dp]
        lib.oracle_scan_bwd.restype = i32
        lib.oracle_scan_bwd.argtypes = [i64, i64, i64, i64, i32, i32,
                                        vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                        dp, dp, dp, i32, vp, i64, dp, dp, dp, dp, dp, dp, dp, dp, dp, i32]
        _lib_cache[path] = lib
    return _lib_cache[path]


def _host(a):
    """(array, type code) for a host array; torch CPU tensors are viewed as numpy."""
    if a is None:
        return None, None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        if a.device.type != "cpu":
            raise ValueError("oracle inputs must be host (CPU) arrays")
        a = a.detach().contiguous()
        if a.dtype == torch.bfloat16:
            return a.view(torch.int16).numpy().view(np.uint16), BF16
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:  # raw bf16 bit patterns
        return a, BF16
    raise TypeError(f"unsupported oracle array dtype {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
             channels=None, h0=None, nthreads: int = 1, lib: ctypes.CDLL | None = None,
             zoh: bool = False):
    """Oracle forward scan.

    Shapes: u, delta, z (batch, dim, L); B, C (batch, L, N); A (dim, N);
    D, delta_bias (dim,).  u/delta/B/C/z share one element type (fp32, bf16
    or fp64); A/D/delta_bias share another (fp32 or fp64).
    ``channels``: optional flat ids b*dim + d to compute (default: all).
    ``h0``: optional fp64 initial state, one row of N per computed channel.
    ``zoh``: the exact zero-order-hold input term (exp(Delta A) - 1) / A B x
    instead of the first-order Delta B x.
    Returns (y, last_state) as fp64 arrays of shape (nchan, L) and (nchan, N);
    with channels=None they are reshaped to (batch, dim, L) and (batch, dim, N).
    """
    lib = lib or load()
    batch, dim, L = (int(s) for s in u.shape)
    N = int(A.shape[1])
    arrs = {}
    for name, a in (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z)):
        arrs[name] = _host(a)
    io_types = {t for _, t in arrs.values() if t is not None}
    if len(io_types) != 1:
        raise TypeError("u, delta, B, C, z must share one element type")
    io = io_types.pop()
    parr = {}
    for name, a in (("A", A), ("D", D), ("bias", delta_bias)):
        parr[name] = _host(a)
    p_types = {t for _, t in parr.values() if t is not None}
    if len(p_types) != 1 or not p_types <= {F32, F64}:
        raise TypeError("A, D, delta_bias must share one element type, fp32 or fp64")
    pio = p_types.pop()
    if channels is None:
        chan = None
        nchan = batch * dim
    else:
        chan = np.ascontiguousarray(np.asarray(channels, dtype=np.int64))
        nchan = int(chan.size)
    y = np.empty((nchan, L), dtype=np.float64)
    last = np.empty((nchan, N), dtype=np.float64)
    if h0 is not None:
        h0 = np.ascontiguousarray(np.asarray(h0, dtype=np.float64).reshape(nchan, N))
    rc = lib.oracle_scan_fwd(batch, dim, N, L, io, pio,
                             _ptr(arrs["u"][0]), _ptr(arrs["delta"][0]), _ptr(parr["A"][0]),
                             _ptr(arrs["B"][0]), _ptr(arrs["C"][0]), _ptr(parr["D"][0]),
                             _ptr(arrs["z"][0]), _ptr(parr["bias"][0]), int(bool(delta_softplus)),
                             int(bool(zoh)), _ptr(chan), nchan, _ptr(h0), _ptr(y), _ptr(last),
                             int(nthreads))
    if rc != 0:
        raise ValueError("oracle_scan_fwd rejected its arguments")
    if channels is None:
        return y.reshape(batch, dim, L), last.reshape(batch, dim, N)
    return y, last


def conv_silu(x, w, conv_bias=None, conv_state=None, lib: ctypes.CDLL | None = None):
    """Oracle short convolution: u = silu(causal depthwise conv(x) + bias).

    x (batch, dim, L) and conv_state (batch, dim, K-1; the inputs before
    token 0, oldest first, or None for zeros) share one element type; w
    (dim, K) and conv_bias (dim,) are fp32 or fp64.  Returns u (batch, dim,
    L) fp64."""
    lib = lib or load()
    batch, dim, L = (int(s) for s in x.shape)
    K = int(w.shape[1])
    xa, xt = _host(x)
    sa, st = _host(conv_state)
    if st is not None and st != xt:
        raise TypeError("x and conv_state must share one element type")
    wa, wt = _host(w)
    ba, bt = _host(conv_bias)
    if wt not in (F32, F64) or (bt is not None and bt != wt):
        raise TypeError("w and conv_bias must share one element type, fp32 or fp64")
    u = np.empty((batch, dim, L), dtype=np.float64)
    rc = lib.oracle_conv_silu(batch, dim, L, K, xt, wt, _ptr(xa), _ptr(wa), _ptr(ba), _ptr(sa),
                              _ptr(u))
    if rc != 0:
        raise ValueError("oracle_conv_silu rejected its arguments")
    return u


def state_step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
               delta_softplus=False, lib: ctypes.CDLL | None = None):
    """Oracle single-token update.  ``state`` (batch, dim, N) fp64 is updated
    in place; returns y (batch, dim) fp64."""
    lib = lib or load()
    if state.dtype != np.float64 or not state.flags["C_CONTIGUOUS"]:
        raise TypeError("oracle state must be a contiguous fp64 array")
    batch, dim, N = (int(s) for s in state.shape)
    arrs = {n: _host(a) for n, a in (("x", x), ("delta", delta), ("B", B), ("C", C), ("z", z))}
    io_types = {t for _, t in arrs.values() if t is not None}
    if len(io_types) != 1:
        raise TypeError("x, delta, B, C, z must share one element type")
    io = io_types.pop()
    parr = {n: _host(a) for n, a in (("A", A), ("D", D), ("bias", delta_bias))}
    p_types = {t for _, t in parr.values() if t is not None}
    if len(p_types) != 1 or not p_types <= {F32, F64}:
        raise TypeError("A, D, delta_bias must share one element type, fp32 or fp64")
    pio = p_types.pop()
    y = np.empty((batch, dim), dtype=np.float64)
    rc = lib.oracle_state_step(batch, dim, N, io, pio, _ptr(state),
                               _ptr(arrs["x"][0]), _ptr(arrs["delta"][0]), _ptr(parr["A"][0]),
                               _ptr(arrs["B"][0]), _ptr(arrs["C"][0]), _ptr(parr["D"][0]),
                               _ptr(arrs["z"][0]), _ptr(parr["bias"][0]),
                               int(bool(delta_softplus)), _ptr(y))
    if rc != 0:
        raise ValueError("oracle_state_step rejected its arguments")
    return y


def scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=False,
             dlast=None, h0=None, channels=None, nthreads: int = 1,
             lib: ctypes.CDLL | None = None, zoh: bool = False):
    """Oracle backward scan: the gradients of a loss with dLoss/dy = ``dy``
    (batch, dim, L) and dLoss/dlast_state = ``dlast`` (batch, dim, N, or
    None) with respect to every input of ``scan_fwd`` run from the initial
    state ``h0`` (batch, dim, N, or None for zero), with the exact
    zero-order-hold input term when ``zoh``.

    Returns a dict of fp64 arrays: du, ddelta, dz (batch, dim, L; dz is None
    without z), dA (dim, N), dD, ddelta_bias (dim,), dB, dC (batch, L, N),
    dh0 (batch, dim, N: the gradient with respect to the initial state).
    The per-channel C code leaves the sums over channels (dB, dC) and over
    the batch (dA, dD, ddelta_bias) to this wrapper.

    ``channels``: flat ids b*dim + d to compute instead of all.  Then the
    result holds the per-channel rows instead of the sums: du, ddelta, dz
    (nchan, L), dA_chan (nchan, N), dD_chan, ddelta_bias_chan (nchan,),
    dh0 (nchan, N); dB, dC are not formed (they need every channel).
    """
    lib = lib or load()
    batch, dim, L = (int(s) for s in u.shape)
    N = int(A.shape[1])
    arrs = {n: _host(a) for n, a in (("u", u), ("delta", delta), ("B", B), ("C", C), ("z", z))}
    io_types = {t for _, t in arrs.values() if t is not None}
    if len(io_types) != 1:
        raise TypeError("u, delta, B, C, z must share one element type")
    io = io_types.pop()
    parr = {n: _host(a) for n, a in (("A", A), ("D", D), ("bias", delta_bias))}
    p_types = {t for _, t in parr.values() if t is not None}
    if len(p_types) != 1 or not p_types <= {F32, F64}:
        raise TypeError("A, D, delta_bias must share one element type, fp32 or fp64")
    pio = p_types.pop()
    dy = np.ascontiguousarray(np.asarray(dy, dtype=np.float64).reshape(batch, dim, L))
    if dlast is not None:
        dlast = np.ascontiguousarray(np.asarray(dlast, dtype=np.float64).reshape(batch, dim, N))
    if h0 is not None:
        h0 = np.ascontiguousarray(np.asarray(h0, dtype=np.float64).reshape(batch, dim, N))
    if channels is None:
        chan, nchan = None, batch * dim
    else:
        chan = np.ascontiguousarray(np.asarray(channels, dtype=np.int64))
        nchan = int(chan.size)
    du = np.empty((nchan, L)); ddelta = np.empty((nchan, L))
    dz = np.empty((nchan, L)) if z is not None else None
    dA = np.empty((nchan, N)); dD = np.empty(nchan); dbias = np.empty(nchan)
    dBc = np.empty((nchan, L, N)); dCc = np.empty((nchan, L, N))
    dh0 = np.empty((nchan, N))
    rc = lib.oracle_scan_bwd(batch, dim, N, L, io, pio,
                             _ptr(arrs["u"][0]), _ptr(arrs["delta"][0]), _ptr(parr["A"][0]),
                             _ptr(arrs["B"][0]), _ptr(arrs["C"][0]), _ptr(parr["D"][0]),
                             _ptr(arrs["z"][0]), _ptr(parr["bias"][0]), int(bool(delta_softplus)),
                             _ptr(dy), _ptr(dlast), _ptr(h0), int(bool(zoh)), _ptr(chan), nchan, _ptr(du),
                             _ptr(ddelta),
                             _ptr(dz), _ptr(dA), _ptr(dD), _ptr(dbias), _ptr(dBc), _ptr(dCc),
                             _ptr(dh0), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_scan_bwd rejected its arguments")
    if channels is not None:
        return {"du": du, "ddelta": ddelta, "dz": dz, "dA_chan": dA, "dD_chan": dD,
                "ddelta_bias_chan": dbias, "dh0": dh0}
    sh = (batch, dim)
    return {"du": du.reshape(*sh, L), "ddelta": ddelta.reshape(*sh, L),
            "dz": None if dz is None else dz.reshape(*sh, L),
            "dA": dA.reshape(*sh, N).sum(axis=0), "dD": dD.reshape(sh).sum(axis=0),
            "ddelta_bias": dbias.reshape(sh).sum(axis=0),
            "dB": dBc.reshape(*sh, L, N).sum(axis=1), "dC": dCc.reshape(*sh, L, N).sum(axis=1),
            "dh0": dh0.reshape(*sh, N)}
