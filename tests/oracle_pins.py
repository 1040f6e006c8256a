"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics.

Each pin takes an oracle library handle (``oracle.load(path)``) so that the
same checks can be re-run against deliberately broken copies of the oracle
(see test_oracle_mutants.py): a plausible mistake anywhere in the oracle
must fail at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from oracle import brute
from scipy.special import expit

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = [float(v) for v in val.split()]
    return out


def close(got, want, rtol, atol=0.0, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {bad.sum()} of {bad.size} off; worst err {err.max():.3e} "
        f"at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def _scalar_scan(lib, delta, u, A=-1.0, h0=None, N=1, extra_A=None, zoh=False):
    """Run the oracle scan with one channel whose state 0 carries the
    scalar recurrence (B=C=1); states 1..N-1, if any, get B=C=0."""
    L = len(delta)
    Bm = np.zeros((1, L, N))
    Cm = np.zeros((1, L, N))
    Bm[0, :, 0] = 1.0
    Cm[0, :, 0] = 1.0
    Am = np.full((1, N), A, np.float64)
    if extra_A is not None and N > 1:
        Am[0, 1:] = extra_A[: N - 1]
    hh = None
    if h0 is not None:
        hh = np.zeros((1, N))
        hh[0, 0] = h0
    y, last = oracle.scan_fwd(np.asarray(u, np.float64)[None, None],
                              np.asarray(delta, np.float64)[None, None],
                              Am, Bm, Cm, channels=[0] if hh is not None else None,
                              h0=hh, lib=lib, zoh=zoh)
    return np.asarray(y).reshape(-1), np.asarray(last).reshape(-1)


# -- pin 1: the one-number gated memory -----------------------------------------
def gate_inputs(gates, xs):
    """Map the page's gate rule h = (1-g) h + g x onto the scan with A = -1,
    B = C = 1: exp(-Delta) = 1 - g gives Delta = -ln(1-g) (g = 1 is taken as
    Delta = 40, where exp(-40) ~ 4e-18), and Delta*u = g*x gives u."""
    deltas, us = [], []
    for g, x in zip(gates, xs):
        if g >= 1.0:
            d = 40.0
        else:
            d = -math.log1p(-g)
        deltas.append(d)
        us.append(g * x / d if d > 0 else x)
    return np.array(deltas), np.array(us)


def pin_gate_fixed(lib):
    gold = read_golden("gate_memory.txt")
    xs = gold["inputs"]
    g = gold["fixed_gate"][0]
    deltas, us = gate_inputs([g] * len(xs), xs)
    for N in (1, 4):
        y, last = _scalar_scan(lib, deltas, us, N=N, extra_A=[-2.0, -3.0, -4.0])
        close(y[:4], gold["fixed_states_first4"], 1e-15, what=f"fixed gate, page values (N={N})")
        # Inputs 2,0,0,0 follow by the same rule: 0.0625/2 + 2/2 = 1.03125, then halving.
        close(y[4:], [1.03125, 0.515625, 0.2578125, 0.12890625], 1e-15,
              what=f"fixed gate, tail (N={N})")
        close(last[0], y[-1], 0.0, what="last_state equals final output")


def pin_gate_selective(lib):
    gold = read_golden("gate_memory.txt")
    deltas, us = gate_inputs(gold["selective_gates"], gold["inputs"])
    for N in (1, 4):
        y, _ = _scalar_scan(lib, deltas, us, N=N, extra_A=[-0.5, -1.5, -7.0])
        close(y, gold["selective_states"], 1e-15, what=f"selective gate (N={N})")


# -- pin 2: affine composition --------------------------------------------------
def pin_affine_compose(lib):
    gold = read_golden("affine_compose.txt")
    (a1, b1), (a2, b2) = gold["first"], gold["second"]
    ca, cb = gold["composed"]
    assert a1 == a2
    dt = -math.log(a1)                       # exp(-dt) = a
    deltas = np.array([dt, dt])
    us = np.array([b1 / dt, b2 / dt])        # dt * u = b
    _, last0 = _scalar_scan(lib, deltas, us)
    close(last0[0], cb, 1e-15, what="composed b (scan from 0)")
    _, last1 = _scalar_scan(lib, deltas, us, h0=1.0)
    close(last1[0] - last0[0], ca, 1e-15, what="composed a (scan, h0 = 1 minus h0 = 0)")
    # the same two updates through the single-token path, from state 1
    state = np.ones((1, 1, 1))
    A = np.full((1, 1), -1.0)
    for d, u in zip(deltas, us):
        oracle.state_step(state, np.array([[u]]), np.array([[d]]), A,
                          np.ones((1, 1)), np.ones((1, 1)), lib=lib)
    close(state[0, 0, 0], ca * 1.0 + cb, 1e-15, what="two state steps from 1")


# -- pin 3: the interactiveml.org scalar zero-order-hold loop -------------------
def page_scalar_loop(inputs, deltas, state=0.0):
    """The page's sequential scalar loop, restated: retention exp(-delta)
    weights the old state and (1 - retention) weights the input."""
    out = []
    for x, d in zip(inputs, deltas):
        retention = math.exp(-d)
        state = retention * state + (1.0 - retention) * x
        out.append(state)
    return np.array(out)


def pin_page_scalar_zoh(lib):
    rng = np.random.default_rng(3)
    L = 500
    x = rng.standard_normal(L)
    d = rng.uniform(0.01, 3.0, L)
    want = page_scalar_loop(x, d)
    # exact ZOH input weight (1 - e^-d) enters the first-order form as u' = x (1 - e^-d)/d
    u = x * (-np.expm1(-d)) / d
    y, last = _scalar_scan(lib, d, u)
    close(y, want, 1e-12, 1e-14, what="page scalar ZOH loop")
    close(last[0], want[-1], 1e-12, what="page scalar ZOH last state")


# -- pin 4: closed form of the constant-step recurrence -------------------------
def pin_closed_form(lib):
    for A, d, L in ((-1.0, 0.25, 1000), (-2.5, 0.01, 3000), (-1.0, 1e-3, 1 << 20)):
        y, last = _scalar_scan(lib, np.full(L, d), np.ones(L), A=A)
        t = np.arange(L)
        # h_t = d * sum_{k=0..t} e^{k A d} = d (1 - e^{(t+1) A d}) / (1 - e^{A d})
        want = d * (-np.expm1((t + 1) * A * d)) / (-math.expm1(A * d))
        close(y, want, 1e-11, what=f"closed form A={A} d={d} L={L}")
        close(last[0], want[-1], 1e-11, what="closed form last state")


# -- pin 5: time-invariant special case equals a convolution ---------------------
def pin_convolution(lib):
    rng = np.random.default_rng(5)
    L, N = 300, 3
    u = rng.standard_normal(L)
    d = 0.3
    A = -np.exp(rng.uniform(0, 1.5, N))
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    Dv = 0.7
    k = np.arange(L)
    K = (Cn[None, :] * np.exp(k[:, None] * d * A[None, :]) * d * Bn[None, :]).sum(1)
    want = np.convolve(u, K)[:L] + Dv * u
    y, _ = oracle.scan_fwd(u[None, None], np.full((1, 1, L), d), A[None],
                           np.tile(Bn, (1, L, 1)), np.tile(Cn, (1, L, 1)),
                           D=np.array([Dv]), lib=lib)
    close(y.reshape(-1), want, 1e-10, 1e-12, what="time-invariant scan vs convolution")


# -- pin 6: brute-force unrolled sum on random tiny inputs ----------------------
def random_tiny(rng, batch, dim, L, N, gate, bias, skip, softplus, dtype=np.float64):
    kw = dict(
        u=rng.standard_normal((batch, dim, L)),
        delta=rng.standard_normal((batch, dim, L)) * 0.8 - (1.0 if softplus else -0.6),
        A=-np.exp(rng.uniform(0, 1.5, (dim, N))),
        B=rng.standard_normal((batch, L, N)),
        C=rng.standard_normal((batch, L, N)),
        D=rng.standard_normal(dim) if skip else None,
        z=rng.standard_normal((batch, dim, L)) * 2 if gate else None,
        delta_bias=rng.uniform(-1, 1, dim) if bias else None,
        delta_softplus=softplus,
    )
    if not softplus:
        kw["delta"] = np.abs(kw["delta"])
    if dtype == np.float64:
        return kw
    out = {}
    for k, v in kw.items():
        if isinstance(v, np.ndarray):
            t = torch.from_numpy(v.astype(np.float32))
            if k in ("A", "D", "delta_bias"):
                out[k] = t                     # parameters stay fp32
            else:
                out[k] = t.to(dtype)
        else:
            out[k] = v
    return out


def _as_f64(kw):
    return {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v) for k, v in kw.items()}


def pin_brute_force(lib):
    rng = np.random.default_rng(6)
    cases = 0
    for gate in (False, True):
        for bias in (False, True):
            for softplus in (False, True):
                for skip in (False, True):
                    L = int(rng.integers(1, 40))
                    N = int(rng.choice([1, 2, 4]))
                    kw = random_tiny(rng, 2, 3, L, N, gate, bias, skip, softplus)
                    y, last = oracle.scan_fwd(**kw, lib=lib)
                    yb, lb = brute.scan_fwd(**kw)
                    close(y, yb, 1e-12, 1e-12, what=f"brute y {gate, bias, softplus, skip}")
                    close(last, lb, 1e-12, 1e-12, what="brute last_state")
                    cases += 1
    # fp32 and bf16 host inputs: the oracle decodes them; brute force gets fp64 copies
    for dt in (torch.float32, torch.bfloat16):
        kw = random_tiny(rng, 2, 5, 33, 4, True, True, True, True, dtype=dt)
        y, last = oracle.scan_fwd(**kw, lib=lib)
        yb, lb = brute.scan_fwd(**_as_f64(kw))
        close(y, yb, 1e-12, 1e-12, what=f"brute y from {dt} inputs")
        close(last, lb, 1e-12, 1e-12, what=f"brute last_state from {dt} inputs")
    assert cases == 16


# -- pin 7: special cases -------------------------------------------------------
def pin_special_cases(lib):
    rng = np.random.default_rng(7)
    kw = random_tiny(rng, 1, 2, 12, 4, False, False, True, False)
    # (a) a zero step freezes the state exactly: exp(0) = 1 and 0 * B * u = 0
    kw["delta"][..., 6:] = 0.0
    _, last_full = oracle.scan_fwd(**kw, lib=lib)
    pre = {k: (v[..., :6] if k in ("u", "delta") else v) for k, v in kw.items()}
    pre["B"] = kw["B"][:, :6]
    pre["C"] = kw["C"][:, :6]
    _, last_pre = oracle.scan_fwd(**pre, lib=lib)
    assert np.array_equal(last_full, last_pre), "zero step must freeze the state"
    # (b) exp(Delta A) underflows to 0: the state forgets everything, h_t = Delta B_t u_t
    kw = random_tiny(rng, 1, 2, 12, 4, False, False, True, False)
    kw["A"] = -np.ones_like(kw["A"])
    kw["delta"] = np.full_like(kw["delta"], 800.0)
    y, last = oracle.scan_fwd(**kw, lib=lib)
    u = kw["u"][0]                                    # (dim, L)
    BC = (kw["B"][0] * kw["C"][0]).sum(-1)            # (L,)
    want = 800.0 * u * BC[None, :] + kw["D"][:, None] * u
    close(y[0], want, 1e-13, 1e-13, what="memoryless limit")
    close(last[0], 800.0 * u[:, -1:] * kw["B"][0, -1][None, :], 1e-13, what="memoryless state")
    # (c) zero input: zero output and zero state, whatever the gate
    kw = random_tiny(rng, 2, 3, 9, 4, True, True, True, True)
    kw["u"] = np.zeros_like(kw["u"])
    y, last = oracle.scan_fwd(**kw, lib=lib)
    assert not y.any() and not last.any(), "u = 0 must give y = 0 and h = 0"
    # (d) empty sequence: no output, state stays at its initial value
    kw = random_tiny(rng, 1, 2, 0, 4, True, False, True, True)
    y, last = oracle.scan_fwd(**kw, lib=lib)
    assert y.shape == (1, 2, 0) and not last.any()


# -- pin 8: recurrent mode equals the scan --------------------------------------
def pin_step_equals_scan(lib):
    rng = np.random.default_rng(8)
    kw = random_tiny(rng, 2, 3, 25, 4, True, True, True, True)
    y, last = oracle.scan_fwd(**kw, lib=lib)
    state = np.zeros((2, 3, 4))
    for t in range(25):
        yt = oracle.state_step(state, kw["u"][..., t].copy(), kw["delta"][..., t].copy(),
                               kw["A"], kw["B"][:, t].copy(), kw["C"][:, t].copy(),
                               D=kw["D"], z=kw["z"][..., t].copy(),
                               delta_bias=kw["delta_bias"], delta_softplus=True, lib=lib)
        close(yt, y[..., t], 1e-14, 1e-14, what=f"step {t} output")
    close(state, last, 1e-14, 1e-14, what="state after all steps")


# -- pin 9: host decoding and channel selection ---------------------------------
def pin_decode_and_subset(lib):
    rng = np.random.default_rng(9)
    kw = random_tiny(rng, 2, 5, 31, 4, True, True, True, True, dtype=torch.bfloat16)
    y, last = oracle.scan_fwd(**kw, lib=lib)
    y64, last64 = oracle.scan_fwd(**_as_f64(kw), lib=lib)
    assert np.array_equal(y, y64) and np.array_equal(last, last64), "bf16 decode must be exact"
    chans = [9, 0, 4, 7]
    ys, ls = oracle.scan_fwd(**kw, channels=chans, lib=lib)
    assert np.array_equal(ys, y.reshape(10, -1)[chans])
    assert np.array_equal(ls, last.reshape(10, -1)[chans])
    yt, lt = oracle.scan_fwd(**kw, nthreads=4, lib=lib)
    assert np.array_equal(yt, y) and np.array_equal(lt, last)


# -- pin 10: the exact zero-order-hold input term -------------------------------
def pin_zoh_page_loop(lib):
    """With the exact input term the scan IS the interactiveml.org scalar
    loop (A = -1, B = C = 1, N = 1), with no input substitution."""
    rng = np.random.default_rng(10)
    L = 500
    x = rng.standard_normal(L)
    d = rng.uniform(0.001, 4.0, L)
    want = page_scalar_loop(x, d)
    y, last = _scalar_scan(lib, d, x, zoh=True)
    close(y, want, 1e-12, 1e-14, what="page scalar loop, exact ZOH")
    close(last[0], want[-1], 1e-12, what="page scalar loop, exact ZOH, last state")
    # and it continues from a given state exactly as the loop does
    y, _ = _scalar_scan(lib, d, x, zoh=True, h0=0.75)
    close(y, page_scalar_loop(x, d, state=0.75), 1e-12, 1e-14, what="page loop from state 0.75")


def pin_zoh_closed_form(lib):
    """Constant step, constant input 1: h_t = B (1 - e^{(t+1) Delta A}) / (-A);
    for A = -1, B = 1 that is the page's 1 - e^{-Delta (t+1)}."""
    for A, d, L in ((-1.0, 0.25, 1000), (-3.0, 0.02, 3000), (-1.0, 1e-3, 1 << 20)):
        y, last = _scalar_scan(lib, np.full(L, d), np.ones(L), A=A, zoh=True)
        t = np.arange(L)
        want = -np.expm1((t + 1) * A * d) / (-A)
        close(y, want, 1e-11, what=f"ZOH closed form A={A} d={d} L={L}")
        close(last[0], want[-1], 1e-11, what="ZOH closed form last state")


def pin_zoh_limits(lib):
    rng = np.random.default_rng(11)
    L = 64
    d = rng.uniform(0.01, 0.5, L)
    u = rng.standard_normal(L)
    # A = 0: (e^{Delta A} - 1) / A -> Delta and e^{Delta A} = 1: a running sum
    y, _ = _scalar_scan(lib, d, u, A=0.0, zoh=True)
    close(y, np.cumsum(d * u), 1e-13, 1e-14, what="ZOH at A = 0: running sum of Delta u")
    # tiny |A|: the exact term agrees with the first-order one to O(Delta A)
    y1, _ = _scalar_scan(lib, d, u, A=-1e-9, zoh=True)
    y0, _ = _scalar_scan(lib, d, u, A=-1e-9, zoh=False)
    close(y1, y0, 1e-8, 1e-12, what="ZOH vs first order as A -> 0")
    # Delta |A| huge: memoryless, h_t = B u_t / (-A)
    y, _ = _scalar_scan(lib, np.full(L, 900.0), u, A=-2.0, zoh=True)
    close(y, u / 2.0, 1e-13, 1e-14, what="ZOH memoryless limit")


def pin_zoh_brute_force(lib):
    rng = np.random.default_rng(12)
    for gate, bias, softplus in ((False, False, False), (True, True, True), (True, False, True)):
        L = int(rng.integers(1, 40))
        kw = random_tiny(rng, 2, 3, L, 4, gate, bias, True, softplus)
        kw["A"][0, 1] = 0.0                  # one state with A = 0 (the limit Delta)
        y, last = oracle.scan_fwd(**kw, zoh=True, lib=lib)
        yb, lb = brute.scan_fwd(**kw, zoh=True)
        close(y, yb, 1e-12, 1e-12, what=f"ZOH brute y {gate, bias, softplus}")
        close(last, lb, 1e-12, 1e-12, what="ZOH brute last_state")


# -- pin 11: the initial state ----------------------------------------------------
def pin_initial_state(lib):
    rng = np.random.default_rng(13)
    for zoh in (False, True):
        kw = random_tiny(rng, 2, 3, 30, 4, True, True, True, True)
        h0 = rng.standard_normal((2, 3, 4))
        # against the unrolled sum, where h0 decays by exp(A_n sum_{r<=t} Delta_r)
        y, last = oracle.scan_fwd(**kw, h0=h0.reshape(6, 4), zoh=zoh, lib=lib)
        yb, lb = brute.scan_fwd(**kw, zoh=zoh, h0=h0)
        close(y, yb, 1e-12, 1e-12, what=f"h0 brute y (zoh={zoh})")
        close(last, lb, 1e-12, 1e-12, what=f"h0 brute last_state (zoh={zoh})")
        # a scan split at k and resumed from its last_state is the whole scan
        k = 11
        head = {n: (v[..., :k] if n in ("u", "delta", "z") else v) for n, v in kw.items()}
        head["B"], head["C"] = kw["B"][:, :k], kw["C"][:, :k]
        tail = {n: (v[..., k:] if n in ("u", "delta", "z") else v) for n, v in kw.items()}
        tail["B"], tail["C"] = kw["B"][:, k:], kw["C"][:, k:]
        yf, lf = oracle.scan_fwd(**kw, zoh=zoh, lib=lib)
        _, lh = oracle.scan_fwd(**head, zoh=zoh, lib=lib)
        yt, lt = oracle.scan_fwd(**tail, h0=lh.reshape(6, 4), zoh=zoh, lib=lib)
        close(yt, yf[..., k:], 1e-12, 1e-13, what=f"split at {k} and resumed, y (zoh={zoh})")
        close(lt, lf, 1e-12, 1e-13, what=f"split at {k} and resumed, last_state (zoh={zoh})")


# -- pin 12: the block's short convolution (causal, depthwise, SiLU) ----------------
def pin_conv_silu(lib):
    rng = np.random.default_rng(14)
    batch, dim, L = 2, 5, 70
    x = rng.standard_normal((batch, dim, L))
    for K in (1, 2, 3, 4):
        w = rng.standard_normal((dim, K))
        cb = rng.standard_normal(dim)
        u = oracle.conv_silu(x, w, conv_bias=cb, lib=lib)
        # against numpy.convolve: output t sees inputs t-K+1 .. t, zeros before 0
        for b in range(batch):
            for d in range(dim):
                pre = np.convolve(x[b, d], w[d, ::-1])[:L] + cb[d]
                close(u[b, d], pre * expit(pre), 1e-13, 1e-14, what=f"conv K={K} ({b},{d})")
        # the impulse response of channel d is its taps, newest tap first, then zeros
        imp = np.zeros((1, dim, L))
        imp[0, :, 10] = 1.0
        ui = oracle.conv_silu(imp, w, lib=lib)
        for d in range(dim):
            pre = np.zeros(L)
            pre[10:10 + K] = w[d, ::-1]
            close(ui[0, d], pre * expit(pre), 1e-14, 1e-15, what=f"impulse response K={K}")
        # a given history continues the sequence: state = the last K-1 inputs
        if K > 1:
            k = 23
            head_state = x[..., k - (K - 1):k].copy()
            ut = oracle.conv_silu(x[..., k:].copy(), w, conv_bias=cb, conv_state=head_state,
                                  lib=lib)
            close(ut, u[..., k:], 1e-14, 1e-15, what=f"conv state continues K={K}")


ALL_PINS = [pin_gate_fixed, pin_gate_selective, pin_affine_compose, pin_page_scalar_zoh,
            pin_closed_form, pin_convolution, pin_brute_force, pin_special_cases,
            pin_step_equals_scan, pin_decode_and_subset, pin_zoh_page_loop,
            pin_zoh_closed_form, pin_zoh_limits, pin_zoh_brute_force, pin_initial_state,
            pin_conv_silu]
