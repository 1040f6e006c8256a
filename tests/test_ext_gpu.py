"""ssm_scan_fwd_ex on the GPU against the fp64 oracle: the exact zero-order-
hold input term, the initial state, and the fused short convolution.

Tolerances are those of parity.py: 1e-4 (1 + |ref|) for fp32 I/O and
2e-2 (1 + |ref|) for bf16 I/O, on y, last_state and the convolution output.
A scan split at token k and resumed from its last_state (and, with the
convolution, from its last K - 1 inputs) runs the same per-token arithmetic
as the whole scan, so those checks are bitwise."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle_pins
import selective_state_space_116_b300 as ssm
from parity import TOL, as64, assert_close, nthreads, to_cuda
from selective_state_space_116_b300.workloads import Workload, make_scan_inputs

pytestmark = pytest.mark.gpu

BASE = Workload("ext", 2, 67, 16, 300, "f32", bias_range=(-4.0, -2.0), a_kind="neg_exp_uniform",
                gate=True)


def f64(t):
    return None if t is None else t.double().numpy()


def gpu_ex(inp, chunk=0, **opts):
    g = to_cuda(inp)
    o = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in opts.items()}
    y, h = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                            delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                            chunk=chunk, check=True, **o)
    torch.cuda.synchronize()
    return y, h


def oracle_ex(inp, zoh=False, h0=None, u=None):
    """The oracle scan; u (fp64) replaces inp["u"] when given (the output of
    the convolution oracle), and then every I/O tensor is passed as fp64."""
    batch, dim, N = inp["u"].shape[0], inp["u"].shape[1], inp["A"].shape[1]
    hh = None if h0 is None else h0.double().numpy().reshape(batch * dim, N)
    if u is None:
        args = dict(u=inp["u"], delta=inp["delta"], B=inp["B"], C=inp["C"], z=inp["z"])
    else:
        args = dict(u=u, delta=f64(inp["delta"]), B=f64(inp["B"]), C=f64(inp["C"]), z=f64(inp["z"]))
    y, h = oracle.scan_fwd(A=inp["A"], D=inp["D"], delta_bias=inp["delta_bias"],
                           delta_softplus=inp["delta_softplus"], zoh=zoh, h0=hh,
                           channels=None if hh is None else np.arange(batch * dim),
                           nthreads=nthreads(), **args)
    return y.reshape(batch, dim, -1), h.reshape(batch, dim, N)


def random_h0(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.batch, w.dim, w.dstate, generator=g) * 2.0


# -- the exact zero-order-hold input term ---------------------------------------
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_zoh_matches_oracle(io, N):
    w = BASE.scaled(io=io, dstate=N)
    inp = make_scan_inputs(w, seed=40 + N)
    y, h = gpu_ex(inp, input_term="zoh")
    y_ref, h_ref = oracle_ex(inp, zoh=True)
    assert_close(as64(y), y_ref, w.torch_io, "zoh y")
    assert_close(as64(h), h_ref, w.torch_io, "zoh last_state")


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("softplus", [False, True])
def test_zoh_options(gate, softplus):
    w = BASE.scaled(gate=gate, softplus=softplus, a_kind="neg_index")
    inp = make_scan_inputs(w, seed=3)
    if not softplus:
        inp["delta"] = inp["delta"].abs() * 0.1
        inp["delta_bias"] = inp["delta_bias"].abs() * 0.01
    y, h = gpu_ex(inp, input_term="zoh")
    y_ref, h_ref = oracle_ex(inp, zoh=True)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


def _scalar(deltas, xs, A=-1.0):
    L = len(deltas)
    f = lambda a: torch.tensor(np.asarray(a, np.float32))
    return {"u": f(xs).reshape(1, 1, L), "delta": f(deltas).reshape(1, 1, L),
            "A": torch.tensor([[A]], dtype=torch.float32), "B": torch.ones(1, L, 1),
            "C": torch.ones(1, L, 1), "D": None, "z": None, "delta_bias": None,
            "delta_softplus": False}


def test_zoh_is_the_page_scalar_loop():
    """With A = -1, B = C = 1 the kernel's exact input term is the
    interactiveml.org loop h = e^-d h + (1 - e^-d) x, step for step, with no
    input substitution; small and large steps both."""
    rng = np.random.default_rng(41)
    L = 2000
    x = rng.standard_normal(L)
    d = np.exp(rng.uniform(np.log(1e-4), np.log(6.0), L))
    want = oracle_pins.page_scalar_loop(x, d)
    inp = _scalar(d, x)
    y, h = gpu_ex(inp, input_term="zoh")
    # the loop's own inputs rounded to fp32 are what the kernel sees
    want32 = oracle_pins.page_scalar_loop(as64(inp["u"]).ravel(), as64(inp["delta"]).ravel())
    assert_close(as64(y).ravel(), want32, torch.float32, "page loop through the kernel")
    assert np.abs(want32 - want).max() < 1e-5


def test_zoh_closed_form():
    """Constant step, constant input 1: h_t = 1 - e^{-Delta (t + 1)}."""
    for d in (0.25, 1e-3, 3.0):
        L = 4096
        inp = _scalar(np.full(L, d), np.ones(L))
        y, _ = gpu_ex(inp, input_term="zoh")
        t = np.arange(L)
        dd = float(np.float32(d))
        assert_close(as64(y).ravel(), -np.expm1(-dd * (t + 1)), torch.float32, f"closed form d={d}")


def test_zoh_at_a_zero():
    """A = 0 for some states: the weight's limit Delta (a running sum of
    Delta u B), next to ordinary decaying states."""
    w = BASE.scaled(dstate=4, a_kind="neg_index")
    inp = make_scan_inputs(w, seed=44)
    A = inp["A"].clone()
    A[:, 1] = 0.0
    A[:, 3] = -1e-7
    inp["A"] = A
    y, h = gpu_ex(inp, input_term="zoh")
    y_ref, h_ref = oracle_ex(inp, zoh=True)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


# -- the initial state -------------------------------------------------------------
@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("zoh", [False, True])
def test_h0_matches_oracle(io, zoh):
    w = BASE.scaled(io=io)
    inp = make_scan_inputs(w, seed=45)
    h0 = random_h0(w, 1)
    y, h = gpu_ex(inp, h0=h0, input_term="zoh" if zoh else "delta_b")
    y_ref, h_ref = oracle_ex(inp, zoh=zoh, h0=h0)
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")


def _split(inp, k):
    head, tail = dict(inp), dict(inp)
    for key in ("u", "delta", "z"):
        if inp[key] is not None:
            head[key] = inp[key][..., :k].contiguous()
            tail[key] = inp[key][..., k:].contiguous()
    for key in ("B", "C"):
        head[key] = inp[key][:, :k].contiguous()
        tail[key] = inp[key][:, k:].contiguous()
    return head, tail


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("N,k", [(4, 96), (16, 131), (16, 1)])
def test_split_and_resume_equals_whole_scan(io, zoh, N, k):
    """A scan over tokens [0, k), then one over [k, L) from its last_state,
    gives the whole scan's outputs bit for bit."""
    w = BASE.scaled(io=io, dstate=N, seqlen=500)
    inp = make_scan_inputs(w, seed=46 + k)
    term = "zoh" if zoh else "delta_b"
    y, h = gpu_ex(inp, input_term=term)
    head, tail = _split(inp, k)
    _, hk = gpu_ex(head, input_term=term)
    yt, ht = gpu_ex(tail, input_term=term, h0=hk)
    assert torch.equal(yt, y[..., k:]) and torch.equal(ht, h)


def test_h0_continued_in_place():
    """h0 may be last_state itself: the state is continued in place."""
    w = BASE.scaled(seqlen=400)
    inp = make_scan_inputs(w, seed=47)
    head, tail = _split(inp, 150)
    _, state = gpu_ex(head)
    g = to_cuda(tail)
    yt, ht = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                              delta_bias=g["delta_bias"], delta_softplus=True, h0=state,
                              last_state=state)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle_ex(inp)
    assert ht.data_ptr() == state.data_ptr()
    assert_close(as64(yt), y_ref[..., 150:], torch.float32, "y")
    assert_close(as64(state), h_ref, torch.float32, "state continued in place")


@pytest.mark.parametrize("chunk", [64, 1300])
def test_h0_and_zoh_through_other_schedules(chunk):
    """The chunked schedule (chunk < L: the first chunk's carry-in is h0) and
    the split persistent schedule (chunk >= L)."""
    w = BASE.scaled(seqlen=1000, dim=130, batch=3)
    inp = make_scan_inputs(w, seed=48)
    h0 = random_h0(w, 2)
    y, h = gpu_ex(inp, chunk=chunk, h0=h0, input_term="zoh")
    y_ref, h_ref = oracle_ex(inp, zoh=True, h0=h0)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


def test_h0_empty_sequence():
    w = BASE.scaled(seqlen=0)
    inp = make_scan_inputs(w)
    h0 = random_h0(w, 3)
    _, h = gpu_ex(inp, h0=h0)
    assert torch.equal(h.cpu(), h0)


# -- the fused short convolution ---------------------------------------------------
def conv_params(w, K, seed, bias=True, state=False):
    g = torch.Generator().manual_seed(seed)
    cw = torch.randn(w.dim, K, generator=g) * 0.5
    cb = torch.randn(w.dim, generator=g) * 0.5 if bias else None
    cs = (torch.randn(w.batch, w.dim, K - 1, generator=g).to(w.torch_io) if state and K > 1
          else None)
    return cw, cb, cs


def oracle_conv(inp, cw, cb, cs):
    return oracle.conv_silu(inp["u"], cw, conv_bias=cb, conv_state=cs)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
def test_conv_matches_oracle(io, K):
    w = BASE.scaled(io=io, seqlen=257)
    inp = make_scan_inputs(w, seed=50 + K)
    cw, cb, cs = conv_params(w, K, K, state=(K == 3))
    u_out = torch.empty(inp["u"].shape, dtype=inp["u"].dtype, device="cuda")
    y, h = gpu_ex(inp, conv_weight=cw, conv_bias=cb, conv_state=cs, u_out=u_out)
    u_ref = oracle_conv(inp, cw, cb, cs)
    y_ref, h_ref = oracle_ex(inp, u=u_ref)
    assert_close(as64(u_out), u_ref, w.torch_io, "convolution output")
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")


@pytest.mark.parametrize("N", [1, 4, 16])
@pytest.mark.parametrize("zoh", [False, True])
def test_conv_with_zoh_and_h0(N, zoh):
    w = BASE.scaled(io="bf16", dstate=N, seqlen=190, dim=70)
    inp = make_scan_inputs(w, seed=55)
    cw, cb, _ = conv_params(w, 4, 6)
    h0 = random_h0(w, 4)
    y, h = gpu_ex(inp, conv_weight=cw, conv_bias=cb, h0=h0, input_term="zoh" if zoh else "delta_b")
    y_ref, h_ref = oracle_ex(inp, zoh=zoh, h0=h0, u=oracle_conv(inp, cw, cb, None))
    assert_close(as64(y), y_ref, torch.bfloat16, "y")
    assert_close(as64(h), h_ref, torch.bfloat16, "last_state")


@pytest.mark.parametrize("chunk", [64, 96, 1300])
def test_conv_through_other_schedules(chunk):
    """Chunks and split groups start mid-sequence: their first tile takes the
    three inputs before it from memory."""
    w = BASE.scaled(seqlen=1000, dim=130, batch=3)
    inp = make_scan_inputs(w, seed=56)
    cw, cb, _ = conv_params(w, 4, 7)
    y, h = gpu_ex(inp, chunk=chunk, conv_weight=cw, conv_bias=cb)
    y_ref, h_ref = oracle_ex(inp, u=oracle_conv(inp, cw, cb, None))
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L,dim", [(1, 3), (7, 64), (33, 65), (1001, 1)])
def test_conv_ragged_shapes(io, L, dim):
    w = BASE.scaled(io=io, seqlen=L, dim=dim, batch=2)
    inp = make_scan_inputs(w, seed=L + dim)
    cw, cb, cs = conv_params(w, 4, 8, state=True)
    u_out = torch.empty(inp["u"].shape, dtype=inp["u"].dtype, device="cuda")
    y, h = gpu_ex(inp, conv_weight=cw, conv_bias=cb, conv_state=cs, u_out=u_out)
    u_ref = oracle_conv(inp, cw, cb, cs)
    y_ref, h_ref = oracle_ex(inp, u=u_ref)
    assert_close(as64(u_out), u_ref, w.torch_io, "convolution output")
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_conv_split_and_resume_equals_whole_scan(io):
    """Resuming needs the state and the last K - 1 inputs: the tail scan with
    h0 = the head's last_state and conv_state = x[k-3 .. k-1] is bitwise the
    whole scan's tail."""
    w = BASE.scaled(io=io, seqlen=600)
    inp = make_scan_inputs(w, seed=57)
    cw, cb, _ = conv_params(w, 4, 9)
    y, h = gpu_ex(inp, conv_weight=cw, conv_bias=cb)
    k = 213
    head, tail = _split(inp, k)
    _, hk = gpu_ex(head, conv_weight=cw, conv_bias=cb)
    cs = inp["u"][..., k - 3:k].contiguous()
    yt, ht = gpu_ex(tail, conv_weight=cw, conv_bias=cb, conv_state=cs, h0=hk)
    assert torch.equal(yt, y[..., k:]) and torch.equal(ht, h)


def test_conv_with_unit_tap_is_silu_of_input():
    """K = 1, tap 1, no bias: u' = silu(x), so the scan equals the plain scan
    on silu(x) -- the fused prologue against the unfused path."""
    w = BASE.scaled(seqlen=300)
    inp = make_scan_inputs(w, seed=58)
    cw = torch.ones(w.dim, 1)
    y, h = gpu_ex(inp, conv_weight=cw)
    plain = dict(inp)
    x = inp["u"].double()
    plain["u"] = (x * torch.sigmoid(x)).float()
    y2, h2 = gpu_ex(plain)
    assert_close(as64(y), as64(y2), torch.float32, "fused vs unfused")
    assert_close(as64(h), as64(h2), torch.float32, "fused vs unfused state")


# -- the configured workload shapes -------------------------------------------------
def _subset(inp, chans):
    """The sub-problem of the listed channels of batch row 0 (batch = 1)."""
    sub = dict(inp)
    idx = torch.from_numpy(np.asarray(chans))
    for key in ("u", "delta", "z"):
        if inp[key] is not None:
            sub[key] = inp[key][:, idx].contiguous()
    sub["A"] = inp["A"][idx].contiguous()
    for key in ("D", "delta_bias"):
        if inp[key] is not None:
            sub[key] = inp[key][idx].contiguous()
    return sub


@pytest.mark.parametrize("name", ["tiny", "m130", "m2p8", "dna"])
@pytest.mark.parametrize("variant", ["zoh_h0", "conv"])
def test_options_on_workload_shapes(name, variant):
    """The exact zero-order hold (with an initial state) and the fused
    convolution at every scan workload's full size; the long DNA-like
    sequence (the chunked schedule) on 64 sampled channels."""
    from selective_state_space_116_b300.workloads import WORKLOADS
    w = WORKLOADS[name]
    inp = make_scan_inputs(w, seed=60)
    if variant == "zoh_h0":
        h0 = random_h0(w, 5)
        opts = dict(input_term="zoh", h0=h0)
    else:
        cw, cb, _ = conv_params(w, 4, 10)
        opts = dict(conv_weight=cw, conv_bias=cb)
    y, h = gpu_ex(inp, **opts)
    if name == "dna":
        chans = np.array(sorted({0, w.dim - 1} | set(np.random.default_rng(3).choice(
            w.dim, 70, replace=False).tolist())))[:64]
        sub = _subset(inp, chans)
        idx = torch.from_numpy(chans).cuda()
        y, h = y[:, idx], h[:, idx]
    else:
        sub = inp
    if variant == "zoh_h0":
        h0s = h0 if name != "dna" else h0[:, torch.from_numpy(chans)].contiguous()
        y_ref, h_ref = oracle_ex(sub, zoh=True, h0=h0s)
    else:
        cws = cw if name != "dna" else cw[torch.from_numpy(chans)].contiguous()
        cbs = cb if name != "dna" else cb[torch.from_numpy(chans)].contiguous()
        y_ref, h_ref = oracle_ex(sub, u=oracle_conv(sub, cws, cbs, None))
    assert_close(as64(y), y_ref, w.torch_io, f"{name} {variant} y")
    assert_close(as64(h), h_ref, w.torch_io, f"{name} {variant} last_state")
