"""Backward scan on the GPU (through the C ABI) against the fp64 backward
oracle (itself pinned by finite differences) on the same seeded inputs.

Tolerance: every gradient is compared in fp64 against the oracle with
|got - ref| <= 1e-3 * max|ref| + 1e-6 over the tensor, and element by
element with |got - ref| <= 2e-3 * |ref| + 1e-4 * max|ref| + 1e-6, so that
the small entries of a tensor (a quiet channel, a token with a small
adjoint) are held to their own size and not only to the largest entry.  The kernel works in fp32 with the
hardware 2^x (relative error ~2^-22); a gradient entry is a sum of up to
L (or batch * L, for dA, dD, ddelta_bias, or dim, for dB, dC) terms, so
its rounding error grows like sqrt(terms) * 2^-23 of the largest term:
below 1e-4 of max|ref| at these sizes, ten times inside the bound."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_116_b300 as ssm
from parity import nthreads, to_cuda
from selective_state_space_116_b300.workloads import WORKLOADS, make_scan_inputs

pytestmark = pytest.mark.gpu

NAMES = ["du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias", "dh0"]


def run_both(w, seed=0, with_dlast=True, with_h0=False, zoh=False, edit=None, chunk=0,
             channels=None):
    inp = make_scan_inputs(w, seed)
    if edit is not None:
        edit(inp)
    rng = np.random.default_rng(seed + 100)
    b, d, L, N = w.batch, w.dim, w.seqlen, w.dstate
    dy = torch.from_numpy(rng.standard_normal((b, d, L)).astype(np.float32))
    dlast = torch.from_numpy(rng.standard_normal((b, d, N)).astype(np.float32)) if with_dlast else None
    h0 = torch.from_numpy((rng.standard_normal((b, d, N)) * 3.0).astype(np.float32)) if with_h0 else None
    g = to_cuda(inp)
    got = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.cuda(), D=g["D"], z=g["z"],
                           delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                           dlast_state=None if dlast is None else dlast.cuda(), return_dh0=True,
                           h0=None if h0 is None else h0.cuda(),
                           input_term="zoh" if zoh else "delta_b", chunk=chunk)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy.double().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"],
                          delta_softplus=inp["delta_softplus"],
                          dlast=None if dlast is None else dlast.double().numpy(),
                          h0=None if h0 is None else h0.double().numpy(), nthreads=nthreads(),
                          zoh=zoh, channels=channels)
    return got, ref


def check(got, ref, what):
    for name in NAMES:
        r, gt = ref[name], got[name]
        if r is None or gt is None:
            assert (gt is None) == (r is None) or name in ("dD", "ddelta_bias"), (what, name)
            continue
        gt = gt.double().cpu().numpy()
        assert gt.shape == r.shape, (what, name, gt.shape, r.shape)
        assert np.all(np.isfinite(gt)), (what, name, "non-finite")
        if r.size == 0:
            continue
        err = np.abs(gt - r)
        scale = np.abs(r).max()
        bound = 1e-3 * scale + 1e-6
        assert err.max() <= bound, f"{what} {name}: max err {err.max():.3e} > {bound:.3e}"
        elem = 2e-3 * np.abs(r) + 1e-4 * scale + 1e-6
        ratio = err / elem
        worst = np.unravel_index(np.argmax(ratio), ratio.shape)
        assert ratio.max() <= 1.0, (f"{what} {name}: {(ratio > 1).sum()} entries outside the "
                                    f"elementwise bound; worst at {worst}: got {gt[worst]:.6g} "
                                    f"ref {r[worst]:.6g}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_bwd_state_sizes(io, N):
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=37, dstate=N, io=io, last_state=True)
    got, ref = run_both(w, seed=N)
    check(got, ref, f"{io} N={N}")


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("L", [40, 64])
def test_bwd_two_channels_per_thread(zoh, L):
    """At N = 16 a grid of at least 1024 two-channel CTAs takes the kernel
    with two channels per thread (smaller grids take one): 4 x 4096
    channels, whole (L = 64) and ragged (L = 40) tiles, from h0, every
    gradient (dB and dC summed over all channels) against the oracle."""
    w = WORKLOADS["m130"].scaled(batch=4, dim=4096, seqlen=L, dstate=16, io="bf16", last_state=True)
    got, ref = run_both(w, seed=L + 3, with_h0=True, zoh=zoh)
    check(got, ref, f"K=2 L={L} zoh={zoh}")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [37, 64])
def test_bwd_from_an_initial_state(io, L):
    """ssm_scan_bwd_ex: the forward ran from h0, so every gradient (dA and
    ddelta through h_(-1), dh0 itself) includes it; L = 64 takes the
    16-byte staging path, L = 37 the element-wise one with a ragged tile."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=L, dstate=16, io=io, last_state=True)
    got, ref = run_both(w, seed=L, with_h0=True)
    check(got, ref, f"{io} L={L} h0")


def zero_and_small_A(inp):
    """A = 0 on one channel and |A| = 1e-3 on another, so that Delta A falls
    on both sides of the kernel's series switches and on their limit."""
    inp["A"][0, :] = 0.0
    inp["A"][1, :] = -1e-3
    inp["A"][2, ::2] = -1e-4


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("L", [37, 64])
def test_bwd_exact_zero_order_hold(io, N, L):
    """ssm_scan_bwd_ex with the exact zero-order-hold input term, from an
    initial state: every gradient against the oracle's (pinned by finite
    differences of the forward oracle with the same term), with A = 0 and
    A near 0 on some channels; L = 64 stages 16 bytes at a time, L = 37 has a
    ragged tile."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=L, dstate=N, io=io, last_state=True)
    got, ref = run_both(w, seed=L + N, with_h0=True, zoh=True, edit=zero_and_small_A)
    check(got, ref, f"{io} N={N} L={L} zoh")


def test_bwd_exact_zero_order_hold_long_sequence():
    """The exact-hold backward over 2048 tokens with softplus(delta) up to
    about 2 (Delta A down to about -30: a = exp(Delta A) underflows to 0 and
    the weight is -1/A), no initial state, against the oracle."""
    w = WORKLOADS["m130"].scaled(batch=1, dim=40, seqlen=2048, dstate=16, io="bf16",
                                 last_state=True, bias_range=(-1.0, 2.0))
    got, ref = run_both(w, seed=5, zoh=True)
    check(got, ref, "zoh L=2048")


def ckpt_bytes(b, d, L, N):
    return b * d * ((L + 7) // 8) * N * 4


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("L,chunk", [(4096, 1024), (4001, 200)])
def test_bwd_chunked(io, N, zoh, L, chunk):
    """The chunked backward (ssm_dims.chunk): chunks of 1024 tokens, where the
    walks for the chunks' maps stop early for most states, and of 200 tokens
    (rounded up to 224: walks over whole chunks) with a ragged last chunk and
    element-wise staging (L = 4001); from h0 with dlast, either input term,
    against the oracle."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=40, seqlen=L, dstate=N, io=io, last_state=True)
    assert (ssm.ssm_scan_bwd_workspace_size(2, 40, N, L, w.torch_io, chunk=chunk) >
            ckpt_bytes(2, 40, L, N))
    got, ref = run_both(w, seed=L + N, with_h0=True, zoh=zoh, chunk=chunk)
    check(got, ref, f"{io} N={N} zoh={zoh} L={L} chunk={chunk}")


@pytest.mark.parametrize("N", [1, 16])
@pytest.mark.parametrize("L,chunk", [(33, 1), (64, 32), (100, 64), (0, 5)])
def test_bwd_chunk_edges(N, L, chunk):
    """Chunks at their smallest: chunk = 1 rounds up to 32, so 33 tokens make
    a 32-token chunk and a 1-token one; two whole 32-token chunks; 64 and 36
    tokens; an empty sequence (one chunk, dh0 = dlast)."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=40, seqlen=L, dstate=N, io="f32", last_state=True)
    got, ref = run_both(w, seed=L + 7, with_h0=True, chunk=chunk)
    check(got, ref, f"N={N} L={L} chunk={chunk}")


def test_bwd_long_sequence_takes_chunks_by_itself():
    """A DNA-like sequence (one-hot inputs, fp32, 2^18 tokens) over 32
    channels: the default schedule cuts it into chunks (its workspace holds
    the chunk arrays).  Per-channel gradients of 8 sampled channels (the
    first and last included) against the oracle; dB and dC, which sum over
    all channels, against the unchunked backward on the GPU."""
    w = WORKLOADS["dna"].scaled(dim=32, seqlen=1 << 18)
    b, d, L, N = w.batch, w.dim, w.seqlen, w.dstate
    assert ssm.ssm_scan_bwd_workspace_size(b, d, N, L, torch.float32) > ckpt_bytes(b, d, L, N)
    assert ssm.ssm_scan_bwd_workspace_size(b, d, N, L, torch.float32, chunk=L) == ckpt_bytes(b, d, L, N)
    chans = [0, 1, 7, 8, 15, 16, 30, 31]
    got, ref = run_both(w, seed=3, channels=chans)
    inp = make_scan_inputs(w, 3)
    rng = np.random.default_rng(103)
    dy = torch.from_numpy(rng.standard_normal((b, d, L)).astype(np.float32))
    dlast = torch.from_numpy(rng.standard_normal((b, d, N)).astype(np.float32))
    g = to_cuda(inp)
    whole = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.cuda(), D=g["D"], z=g["z"],
                             delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                             dlast_state=dlast.cuda(), chunk=L)
    for name in ("du", "ddelta", "dh0"):
        gt = got[name].reshape(b * d, -1)[chans].double().cpu().numpy()
        r = ref[name]
        err = np.abs(gt - r)
        assert err.max() <= 1e-3 * np.abs(r).max() + 1e-6, (name, err.max())
        assert np.all(err <= 2e-3 * np.abs(r) + 1e-4 * np.abs(r).max() + 1e-6), name
    for name, gname in (("dA_chan", "dA"), ("dD_chan", "dD")):
        gt = got[gname][chans].double().cpu().numpy()
        r = ref[name]
        assert np.abs(gt - r).max() <= 1e-3 * np.abs(r).max() + 1e-6, gname
    for name in ("dB", "dC"):
        gt, r = got[name].double().cpu().numpy(), whole[name].double().cpu().numpy()
        err = np.abs(gt - r)
        assert err.max() <= 1e-3 * np.abs(r).max() + 1e-6, (name, err.max())


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("L,chunk", [(64, 0), (37, 0), (4096, 1024)])
def test_bwd_gradients_in_the_io_type(zoh, L, chunk):
    """grad_dtype = bf16: dy read in bf16 gives the fp32 path's gradients for
    the same dy values, and du, ddelta, dz written in bf16 are those fp32
    results rounded to nearest even, bit for bit (16-byte staging at L = 64,
    element-wise at L = 37, chunks at L = 4096); the fp32-only gradients
    agree up to the atomics' order."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=L, io="bf16", last_state=True)
    g = to_cuda(make_scan_inputs(w, seed=L))
    rng = np.random.default_rng(L)
    dy = torch.from_numpy(rng.standard_normal((2, 70, L)).astype(np.float32)).cuda().to(torch.bfloat16)
    kw = dict(D=g["D"], z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True,
              input_term="zoh" if zoh else "delta_b", chunk=chunk)
    full = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.float(), **kw)
    half = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, grad_dtype=torch.bfloat16, **kw)
    for name in ("du", "ddelta", "dz"):
        assert half[name].dtype == torch.bfloat16
        assert torch.equal(half[name], full[name].to(torch.bfloat16)), name
    for name in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        assert half[name].dtype == torch.float32
        r = full[name]
        assert (half[name] - r).abs().max() <= 1e-5 * r.abs().max() + 1e-6, name
    with pytest.raises(TypeError):
        ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, grad_dtype=torch.float16, **kw)
    with pytest.raises(TypeError):   # dy must have the gradient dtype
        ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.float(),
                         grad_dtype=torch.bfloat16, **kw)


def test_bwd_rejects_an_unknown_input_term():
    w = WORKLOADS["m130"].scaled(batch=1, dim=8, seqlen=16, dstate=4, io="f32")
    g = to_cuda(make_scan_inputs(w, 0))
    dy = torch.zeros((1, 8, 16), device="cuda")
    with pytest.raises(ValueError):
        ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, input_term="exact")


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("softplus", [False, True])
@pytest.mark.parametrize("extras", [False, True])
def test_bwd_options(gate, softplus, extras):
    w = WORKLOADS["m130"].scaled(batch=2, dim=33, seqlen=50, io="f32", gate=gate,
                                 softplus=softplus, last_state=True,
                                 bias_range=(((-4.0, -2.0) if softplus else (0.1, 0.5))
                                             if extras else None))
    inp = make_scan_inputs(w, seed=7)
    if not extras:
        inp["D"] = None
    if not softplus:
        inp["delta"] = inp["delta"].abs()
    rng = np.random.default_rng(9)
    dy = torch.from_numpy(rng.standard_normal((2, 33, 50)).astype(np.float32))
    g = to_cuda(inp)
    got = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.cuda(), D=g["D"], z=g["z"],
                           delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                           return_dh0=True)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy.double().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"],
                          delta_softplus=inp["delta_softplus"])
    check(got, ref, f"gate={gate} softplus={softplus} extras={extras}")


@pytest.mark.parametrize("L", [1, 8, 9, 300])
def test_bwd_lengths_and_ragged_channels(L):
    w = WORKLOADS["m130"].scaled(batch=3, dim=130, seqlen=L, last_state=True)
    got, ref = run_both(w, seed=L)
    check(got, ref, f"L={L}")


def test_bwd_layer_shape_m2p8_sampled_channels():
    """The Mamba-2.8B layer shape at full size: every per-channel gradient
    (du, ddelta, dz, dh0) of sampled channels, and dA, dD, ddelta_bias of the
    sampled channels (summed over all batch rows), against the oracle run on
    those channels only.  dB and dC sum over all 5120 channels and are
    covered by the smaller shapes above."""
    w = WORKLOADS["m2p8"]
    inp = make_scan_inputs(w, seed=0)
    rng = np.random.default_rng(42)
    dy = torch.from_numpy(rng.standard_normal((w.batch, w.dim, w.seqlen)).astype(np.float32))
    g = to_cuda(inp)
    got = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy.cuda(), D=g["D"], z=g["z"],
                           delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                           return_dh0=True)
    torch.cuda.synchronize()
    ds = sorted({0, 1, 63, 64, 2559, w.dim - 1, *rng.choice(w.dim, 4, replace=False).tolist()})
    chans = [b * w.dim + d for d in ds for b in range(w.batch)]
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], dy.double().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"],
                          delta_softplus=inp["delta_softplus"], channels=chans, nthreads=nthreads())
    flat = {k: got[k].reshape(w.batch * w.dim, -1) for k in ("du", "ddelta", "dz", "dh0")}
    for name in ("du", "ddelta", "dz", "dh0"):
        r = ref[name]
        gt = flat[name][chans].double().cpu().numpy()
        err = np.abs(gt - r).max()
        assert err <= 1e-3 * np.abs(r).max() + 1e-6, (name, err)
    for name, gname in (("dA_chan", "dA"), ("dD_chan", "dD"), ("ddelta_bias_chan", "ddelta_bias")):
        r = ref[name].reshape(len(ds), w.batch, *ref[name].shape[1:]).sum(axis=1)
        gt = got[gname][ds].double().cpu().numpy()
        err = np.abs(gt - r).max()
        assert err <= 1e-3 * np.abs(r).max() + 1e-6, (gname, err)


def test_autograd_wrapper_with_initial_state():
    """selective_scan(h0=...): the forward starts from h0 (equal to
    ssm_scan_fwd's) and h0 gets its gradient, matching the oracle."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=45, io="f32", last_state=True)
    inp = make_scan_inputs(w, seed=6)
    g = to_cuda(inp)
    rng = np.random.default_rng(9)
    h0 = torch.from_numpy(rng.standard_normal((w.batch, w.dim, w.dstate)).astype(np.float32)).cuda()
    leaves = {k: g[k].clone().requires_grad_(True) for k in ("u", "A")}
    h0l = h0.clone().requires_grad_(True)
    y, last = ssm.selective_scan(leaves["u"], g["delta"], leaves["A"], g["B"], g["C"], D=g["D"],
                                 z=g["z"], delta_bias=g["delta_bias"], delta_softplus=True, h0=h0l)
    y_ref, last_ref = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                       delta_bias=g["delta_bias"], delta_softplus=True, h0=h0)
    assert torch.equal(y.detach(), y_ref) and torch.equal(last.detach(), last_ref)
    wy = torch.from_numpy(rng.standard_normal(tuple(y.shape)).astype(np.float32)).cuda()
    wl = torch.from_numpy(rng.standard_normal(tuple(last.shape)).astype(np.float32)).cuda()
    ((y * wy).sum() + (last * wl).sum()).backward()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], wy.double().cpu().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"], delta_softplus=True,
                          dlast=wl.double().cpu().numpy(), h0=h0.double().cpu().numpy())
    for gt, r, name in ((leaves["u"].grad, ref["du"], "du"), (leaves["A"].grad, ref["dA"], "dA"),
                        (h0l.grad, ref["dh0"], "dh0")):
        gt = gt.double().cpu().numpy()
        assert gt.shape == r.shape, (name, gt.shape, r.shape)
        err = np.abs(gt - r).max()
        assert err <= 1e-3 * np.abs(r).max() + 1e-6, (name, err)


def test_autograd_wrapper_exact_zero_order_hold():
    """selective_scan(input_term="zoh"): the forward equals ssm_scan_fwd's
    with the same term bit for bit, and every gradient matches the oracle's
    backward of the exact-hold recurrence."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=45, io="f32", last_state=True)
    inp = make_scan_inputs(w, seed=12)
    zero_and_small_A(inp)
    g = to_cuda(inp)
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
    leaves = {k: g[k].clone().requires_grad_(True) for k in names}
    y, last = ssm.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                                 D=leaves["D"], z=leaves["z"], delta_bias=leaves["delta_bias"],
                                 delta_softplus=True, input_term="zoh")
    y_ref, last_ref = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                       delta_bias=g["delta_bias"], delta_softplus=True,
                                       return_last_state=True, input_term="zoh")
    assert torch.equal(y.detach(), y_ref) and torch.equal(last.detach(), last_ref)
    rng = np.random.default_rng(13)
    wy = torch.from_numpy(rng.standard_normal(tuple(y.shape)).astype(np.float32)).cuda()
    wl = torch.from_numpy(rng.standard_normal(tuple(last.shape)).astype(np.float32)).cuda()
    ((y * wy).sum() + (last * wl).sum()).backward()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], wy.double().cpu().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"], delta_softplus=True,
                          dlast=wl.double().cpu().numpy(), zoh=True)
    for k, rk in (("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("D", "dD"),
                  ("z", "dz"), ("delta_bias", "ddelta_bias")):
        gt = leaves[k].grad.double().cpu().numpy()
        r = ref[rk]
        assert gt.shape == r.shape, (k, gt.shape, r.shape)
        err = np.abs(gt - r).max()
        assert err <= 1e-3 * np.abs(r).max() + 1e-6, (k, err)


def test_autograd_wrapper_bf16_gradients():
    """selective_scan on bf16 inputs: the backward takes the bf16 upstream
    gradient as it is and returns du, ddelta, dz in bf16, equal bit for bit
    to ssm_scan_bwd's fp32 gradients for the same upstream values rounded
    once; dA, dB, dC, dD, ddelta_bias as ssm_scan_bwd gives them (cast to
    the inputs' dtype), up to the atomics' order."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=64, io="bf16", last_state=True)
    g = to_cuda(make_scan_inputs(w, seed=21))
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
    leaves = {k: g[k].clone().requires_grad_(True) for k in names}
    y, last = ssm.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                                 D=leaves["D"], z=leaves["z"], delta_bias=leaves["delta_bias"],
                                 delta_softplus=True)
    rng = np.random.default_rng(22)
    wy = torch.from_numpy(rng.standard_normal(tuple(y.shape)).astype(np.float32)).cuda().to(torch.bfloat16)
    wl = torch.from_numpy(rng.standard_normal(tuple(last.shape)).astype(np.float32)).cuda()
    torch.autograd.backward((y, last), (wy, wl))
    ref = ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], wy.float(), D=g["D"], z=g["z"],
                           delta_bias=g["delta_bias"], delta_softplus=True, dlast_state=wl)
    for k, rk in (("u", "du"), ("delta", "ddelta"), ("z", "dz")):
        assert leaves[k].grad.dtype == torch.bfloat16, k
        assert torch.equal(leaves[k].grad, ref[rk].to(torch.bfloat16)), k
    for k, rk in (("A", "dA"), ("B", "dB"), ("C", "dC"), ("D", "dD"), ("delta_bias", "ddelta_bias")):
        got, r = leaves[k].grad.float(), ref[rk].to(leaves[k].dtype).float()
        assert (got - r).abs().max() <= 1e-2 * r.abs().max() + 1e-6, k


def test_autograd_wrapper_returns_the_library_gradients():
    """selective_scan under torch.autograd: the forward equals ssm_scan_fwd
    bit for bit and the gradients equal ssm_scan_bwd's for the same upstream
    gradient (up to the fp32 atomics' summation order for dA, dB, dC, dD,
    ddelta_bias), and they match the oracle."""
    w = WORKLOADS["m130"].scaled(batch=2, dim=70, seqlen=45, io="f32", last_state=True)
    inp = make_scan_inputs(w, seed=4)
    g = to_cuda(inp)
    leaves = {k: g[k].clone().requires_grad_(True) for k in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    y, last = ssm.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                                 D=leaves["D"], z=leaves["z"], delta_bias=leaves["delta_bias"],
                                 delta_softplus=True)
    y_ref, last_ref = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                                       delta_bias=g["delta_bias"], delta_softplus=True)
    assert torch.equal(y.detach(), y_ref) and torch.equal(last.detach(), last_ref)
    rng = np.random.default_rng(8)
    wy = torch.from_numpy(rng.standard_normal(tuple(y.shape)).astype(np.float32)).cuda()
    wl = torch.from_numpy(rng.standard_normal(tuple(last.shape)).astype(np.float32)).cuda()
    ((y * wy).sum() + (last * wl).sum()).backward()
    ref = oracle.scan_bwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], wy.double().cpu().numpy(),
                          D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"], delta_softplus=True,
                          dlast=wl.double().cpu().numpy())
    for k, rk in (("u", "du"), ("delta", "ddelta"), ("A", "dA"), ("B", "dB"), ("C", "dC"), ("D", "dD"),
                  ("z", "dz"), ("delta_bias", "ddelta_bias")):
        gt = leaves[k].grad.double().cpu().numpy()
        r = ref[rk]
        assert gt.shape == r.shape, (k, gt.shape, r.shape)
        err = np.abs(gt - r).max()
        assert err <= 1e-3 * np.abs(r).max() + 1e-6, (k, err)
