"""Pins for the backward oracle: every gradient it returns must equal the
central finite difference of the forward oracle (fp64) for the scalar loss
sum(y * Wy) + sum(last_state * Wh), on tiny random inputs, with and without
each option.  The derivative's definition is the reference here; nothing in
the backward code is reused."""
import numpy as np
import pytest

import oracle

EPS = 1e-6
RTOL = 1e-6


def make(rng, b, d, L, N, z, softplus, bias, skip):
    x = dict(
        u=rng.standard_normal((b, d, L)),
        delta=rng.standard_normal((b, d, L)) * 0.5 + (0.0 if softplus else 1.0),
        A=-np.exp(rng.uniform(0.0, 1.5, (d, N))),
        B=rng.standard_normal((b, L, N)),
        C=rng.standard_normal((b, L, N)),
        D=rng.standard_normal(d) if skip else None,
        z=rng.standard_normal((b, d, L)) if z else None,
        delta_bias=rng.uniform(-1.0, 0.5, d) if bias else None,
    )
    if not softplus:
        x["delta"] = np.abs(x["delta"])
    return x


def loss(x, softplus, Wy, Wh, h0=None, zoh=False):
    y, h = oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                           delta_bias=x["delta_bias"], delta_softplus=softplus, h0=h0, zoh=zoh)
    return float((y * Wy).sum() + (h * Wh).sum())


@pytest.mark.parametrize("opts", [
    dict(z=True, softplus=True, bias=True, skip=True),
    dict(z=False, softplus=False, bias=False, skip=False),
    dict(z=True, softplus=False, bias=True, skip=False),
    dict(z=False, softplus=True, bias=False, skip=True),
])
@pytest.mark.parametrize("shape", [(2, 3, 7, 4), (1, 2, 1, 1), (1, 1, 13, 2)])
def test_backward_oracle_matches_finite_differences(opts, shape):
    b, d, L, N = shape
    rng = np.random.default_rng(11)
    x = make(rng, b, d, L, N, **opts)
    sp = opts["softplus"]
    Wy = rng.standard_normal((b, d, L))
    Wh = rng.standard_normal((b, d, N))
    g = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], Wy, D=x["D"], z=x["z"],
                        delta_bias=x["delta_bias"], delta_softplus=sp, dlast=Wh)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    for name, gname in names.items():
        if x[name] is None:
            continue
        arr = x[name]
        an = g[gname]
        assert an.shape == arr.shape, (name, an.shape, arr.shape)
        flat = arr.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 12), replace=False)
        for i in idx:
            keep = flat[i]
            flat[i] = keep + EPS
            lp = loss(x, sp, Wy, Wh)
            flat[i] = keep - EPS
            lm = loss(x, sp, Wy, Wh)
            flat[i] = keep
            fd = (lp - lm) / (2 * EPS)
            got = an.reshape(-1)[i]
            assert abs(fd - got) <= RTOL * (1 + abs(fd)), (name, int(i), fd, got)
    # gradient with respect to the initial state, through scan_fwd's h0
    h0 = np.zeros((b * d, N))
    for i in rng.choice(h0.size, size=min(h0.size, 6), replace=False):
        hp = h0.copy(); hp.reshape(-1)[i] += EPS
        hm = h0.copy(); hm.reshape(-1)[i] -= EPS
        fd = (loss(x, sp, Wy, Wh, hp) - loss(x, sp, Wy, Wh, hm)) / (2 * EPS)
        got = g["dh0"].reshape(-1)[i]
        assert abs(fd - got) <= RTOL * (1 + abs(fd)), ("h0", int(i), fd, got)


@pytest.mark.parametrize("opts", [
    dict(z=True, softplus=True, bias=True, skip=True),
    dict(z=False, softplus=False, bias=False, skip=False),
])
def test_backward_oracle_with_initial_state_matches_finite_differences(opts):
    """The forward run from a nonzero initial state h0: every gradient,
    including dh0 around that h0 and the dA, dDelta terms that h0 feeds
    through h_(-1), against central differences of the forward oracle."""
    b, d, L, N = 2, 3, 9, 4
    rng = np.random.default_rng(23)
    x = make(rng, b, d, L, N, **opts)
    sp = opts["softplus"]
    Wy = rng.standard_normal((b, d, L))
    Wh = rng.standard_normal((b, d, N))
    h0 = rng.standard_normal((b * d, N)) * 2.0
    g = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], Wy, D=x["D"], z=x["z"],
                        delta_bias=x["delta_bias"], delta_softplus=sp, dlast=Wh,
                        h0=h0.reshape(b, d, N))
    g0 = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], Wy, D=x["D"], z=x["z"],
                         delta_bias=x["delta_bias"], delta_softplus=sp, dlast=Wh)
    assert not np.allclose(g["dA"], g0["dA"])   # h0 reaches dA
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    for name, gname in names.items():
        if x[name] is None:
            continue
        flat = x[name].reshape(-1)
        for i in rng.choice(flat.size, size=min(flat.size, 10), replace=False):
            keep = flat[i]
            flat[i] = keep + EPS
            lp = loss(x, sp, Wy, Wh, h0)
            flat[i] = keep - EPS
            lm = loss(x, sp, Wy, Wh, h0)
            flat[i] = keep
            fd = (lp - lm) / (2 * EPS)
            got = g[gname].reshape(-1)[i]
            assert abs(fd - got) <= RTOL * (1 + abs(fd)), (name, int(i), fd, got)
    for i in rng.choice(h0.size, size=8, replace=False):
        hp = h0.copy(); hp.reshape(-1)[i] += EPS
        hm = h0.copy(); hm.reshape(-1)[i] -= EPS
        fd = (loss(x, sp, Wy, Wh, hp) - loss(x, sp, Wy, Wh, hm)) / (2 * EPS)
        got = g["dh0"].reshape(-1)[i]
        assert abs(fd - got) <= RTOL * (1 + abs(fd)), ("h0", int(i), fd, got)


@pytest.mark.parametrize("opts", [
    dict(z=True, softplus=True, bias=True, skip=True),
    dict(z=False, softplus=False, bias=False, skip=True),
])
@pytest.mark.parametrize("with_h0", [False, True])
def test_backward_oracle_exact_hold_matches_finite_differences(opts, with_h0):
    """The exact zero-order-hold input term ((exp(Delta A) - 1) / A B u): every
    gradient against central differences of the forward oracle.  Some A are
    0 and some -1e-3 (|Delta A| below the series switch of dw/dA), the rest
    ordinary, so dA is checked on both sides of the switch and at A = 0."""
    b, d, L, N = 2, 3, 8, 4
    rng = np.random.default_rng(31)
    x = make(rng, b, d, L, N, **opts)
    x["A"][0, 0] = 0.0
    x["A"][1, 1] = -1e-3
    x["A"][2, 2] = -1.0 / 16
    sp = opts["softplus"]
    Wy = rng.standard_normal((b, d, L))
    Wh = rng.standard_normal((b, d, N))
    h0 = rng.standard_normal((b * d, N)) if with_h0 else None
    g = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], Wy, D=x["D"], z=x["z"],
                        delta_bias=x["delta_bias"], delta_softplus=sp, dlast=Wh,
                        h0=None if h0 is None else h0.reshape(b, d, N), zoh=True)
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    for name, gname in names.items():
        if x[name] is None:
            continue
        flat = x[name].reshape(-1)
        idx = np.arange(flat.size) if name == "A" else \
            rng.choice(flat.size, size=min(flat.size, 10), replace=False)
        for i in idx:
            keep = flat[i]
            flat[i] = keep + EPS
            lp = loss(x, sp, Wy, Wh, h0, zoh=True)
            flat[i] = keep - EPS
            lm = loss(x, sp, Wy, Wh, h0, zoh=True)
            flat[i] = keep
            fd = (lp - lm) / (2 * EPS)
            got = g[gname].reshape(-1)[i]
            assert abs(fd - got) <= RTOL * (1 + abs(fd)), (name, int(i), fd, got)
    hb = np.zeros((b * d, N)) if h0 is None else h0
    for i in rng.choice(hb.size, size=6, replace=False):
        hp = hb.copy(); hp.reshape(-1)[i] += EPS
        hm = hb.copy(); hm.reshape(-1)[i] -= EPS
        fd = (loss(x, sp, Wy, Wh, hp, zoh=True) - loss(x, sp, Wy, Wh, hm, zoh=True)) / (2 * EPS)
        got = g["dh0"].reshape(-1)[i]
        assert abs(fd - got) <= RTOL * (1 + abs(fd)), ("h0", int(i), fd, got)


def test_backward_oracle_zero_gradient_and_linearity():
    rng = np.random.default_rng(3)
    x = make(rng, 2, 2, 9, 4, z=False, softplus=True, bias=True, skip=True)
    zero = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], np.zeros((2, 2, 9)),
                           D=x["D"], delta_bias=x["delta_bias"], delta_softplus=True)
    for k, v in zero.items():
        if v is not None:
            assert np.all(v == 0.0), k
    # the gradient is linear in dy
    dy1, dy2 = rng.standard_normal((2, 2, 9)), rng.standard_normal((2, 2, 9))
    run = lambda dy: oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x["D"],
                                     delta_bias=x["delta_bias"], delta_softplus=True)
    g1, g2, g12 = run(dy1), run(dy2), run(dy1 + 2.0 * dy2)
    for k in g1:
        if g1[k] is not None:
            np.testing.assert_allclose(g12[k], g1[k] + 2.0 * g2[k], rtol=1e-10, atol=1e-12)


def test_backward_oracle_channel_subset_matches_full():
    """A channel subset gives exactly the full computation's per-channel rows,
    and the per-channel shares sum to the full dA, dD, ddelta_bias."""
    rng = np.random.default_rng(5)
    b, d, L, N = 3, 5, 11, 4
    x = make(rng, b, d, L, N, z=True, softplus=True, bias=True, skip=True)
    dy = rng.standard_normal((b, d, L))
    dl = rng.standard_normal((b, d, N))
    full = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x["D"], z=x["z"],
                           delta_bias=x["delta_bias"], delta_softplus=True, dlast=dl)
    chans = [0, 7, 14, 3]
    sub = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x["D"], z=x["z"],
                          delta_bias=x["delta_bias"], delta_softplus=True, dlast=dl, channels=chans)
    for k, c in enumerate(chans):
        bb, dd = divmod(c, d)
        for name in ("du", "ddelta", "dz", "dh0"):
            assert np.array_equal(sub[name][k], full[name][bb, dd]), name
    allc = oracle.scan_bwd(x["u"], x["delta"], x["A"], x["B"], x["C"], dy, D=x["D"], z=x["z"],
                           delta_bias=x["delta_bias"], delta_softplus=True, dlast=dl,
                           channels=list(range(b * d)))
    np.testing.assert_allclose(allc["dA_chan"].reshape(b, d, N).sum(0), full["dA"], rtol=1e-14)
    np.testing.assert_allclose(allc["dD_chan"].reshape(b, d).sum(0), full["dD"], rtol=1e-14)
    np.testing.assert_allclose(allc["ddelta_bias_chan"].reshape(b, d).sum(0), full["ddelta_bias"],
                               rtol=1e-14)
