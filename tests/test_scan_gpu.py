"""Forward-scan parity: the CUDA library (through its C ABI) against the fp64
oracle on the same seeded inputs.  Tolerances are stated in parity.py:
1e-4*(1+|ref|) for fp32 I/O, 2e-2*(1+|ref|) for bf16 I/O, on y and last_state."""
import math

import numpy as np
import pytest
import torch

import oracle_pins
from parity import TOL, as64, assert_close, gpu_scan, oracle_scan, sample_channels
from selective_state_space_116_b300.workloads import WORKLOADS, Workload, make_scan_inputs

pytestmark = pytest.mark.gpu


def check_full(w: Workload, seed=0, chunk=0):
    inp = make_scan_inputs(w, seed)
    y, h = gpu_scan(inp, chunk=chunk)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, w.torch_io, f"{w.name} y")
    assert_close(as64(h), h_ref, w.torch_io, f"{w.name} last_state")
    return inp, y, h


def test_tiny_workload():
    check_full(WORKLOADS["tiny"])


# small shapes that span several channel blocks and token tiles plus ragged tails
BASE = Workload("opt", 2, 67, 16, 131, "bf16", bias_range=(-4.0, -2.0), a_kind="neg_index",
                gate=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_state_sizes(io, N):
    check_full(BASE.scaled(io=io, dstate=N, a_kind="neg_exp_uniform"), seed=N)


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("softplus", [False, True])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("skip", [False, True])
def test_options(gate, softplus, bias, skip):
    w = BASE.scaled(io="f32", gate=gate, softplus=softplus, skip=skip,
                    bias_range=(-4.0, -2.0) if bias else None,
                    delta_mean=0.0 if softplus else 0.0)
    inp = make_scan_inputs(w, seed=11)
    if not softplus:  # a positive step size without softplus
        inp["delta"] = inp["delta"].abs() * 0.1
        if inp["delta_bias"] is not None:
            inp["delta_bias"] = inp["delta_bias"].abs() * 0.01
    y, h = gpu_scan(inp)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [1, 7, 63, 64, 65, 256, 1000])
@pytest.mark.parametrize("dim", [1, 3, 64, 130])
def test_ragged_shapes(io, L, dim):
    check_full(BASE.scaled(io=io, dim=dim, seqlen=L, batch=1 if dim > 64 else 3), seed=L + dim)


def test_empty_sequence():
    w = BASE.scaled(seqlen=0)
    inp = make_scan_inputs(w)
    y, h = gpu_scan(inp)
    assert y.shape == (2, 67, 0)
    assert torch.count_nonzero(h).item() == 0


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("bias", [-12.0, -18.0, -40.0])
def test_softplus_of_strongly_negative_inputs(io, bias):
    """delta + bias far below zero: softplus(v) ~ e^v is tiny, where
    ln(1 + e^v) formed in fp32 would lose most of its bits (at v = -18,
    1 + e^v rounds to 1 and the step size would vanish)."""
    w = BASE.scaled(io=io, gate=False, skip=False, bias_range=(bias, bias + 1e-3), seqlen=300)
    inp = make_scan_inputs(w, seed=21)
    y, h = gpu_scan(inp)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")
    # With u scaled by e^-bias the states are O(100) and every input term
    # is proportional to its Delta, so a relative error in Delta shows as the
    # same relative error in the states.  Bound the largest error by 1e-5
    # (fp32) or 2e-3 (bf16) of the largest state: fp32 rounding of the sums
    # stays near 1e-6 of it, while the error of ln(1 + e^v) formed in fp32
    # (0.5% at v = -12, the whole step size at v = -18) is far above.
    big = dict(inp)
    big["u"] = (inp["u"].float() * float(np.exp(-bias))).to(inp["u"].dtype)
    _, h = gpu_scan(big)
    _, h_ref = oracle_scan(big)
    scale = np.abs(h_ref).max()
    assert scale > 50.0
    err = np.abs(as64(h) - h_ref).max()
    assert err <= (1e-5 if io == "f32" else 2e-3) * scale, (err, scale)


def test_without_last_state():
    w = BASE.scaled(io="bf16")
    inp = make_scan_inputs(w, seed=5)
    y, h = gpu_scan(inp, return_last_state=False)
    assert h is None
    y_ref, _ = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.bfloat16, "y")


# -- the pages' worked examples, run through the CUDA kernel --------------------
def _scalar_inputs(deltas, us, h_A=-1.0):
    L = len(deltas)
    f = lambda a: torch.tensor(np.asarray(a, np.float32))
    return {
        "u": f(us).reshape(1, 1, L), "delta": f(deltas).reshape(1, 1, L),
        "A": torch.tensor([[h_A]], dtype=torch.float32),
        "B": torch.ones(1, L, 1), "C": torch.ones(1, L, 1), "D": None, "z": None,
        "delta_bias": None, "delta_softplus": False,
    }


def test_gate_example_on_gpu():
    gold = oracle_pins.read_golden("gate_memory.txt")
    xs = gold["inputs"]
    d, u = oracle_pins.gate_inputs([gold["fixed_gate"][0]] * len(xs), xs)
    y, _ = gpu_scan(_scalar_inputs(d, u))
    assert_close(as64(y).reshape(-1)[:4], gold["fixed_states_first4"], torch.float32, "fixed")
    d, u = oracle_pins.gate_inputs(gold["selective_gates"], xs)
    y, _ = gpu_scan(_scalar_inputs(d, u))
    assert_close(as64(y).reshape(-1), gold["selective_states"], torch.float32, "selective")


def test_affine_compose_on_gpu():
    gold = oracle_pins.read_golden("affine_compose.txt")
    (a1, b1), (_, b2) = gold["first"], gold["second"]
    dt = -math.log(a1)
    y, h = gpu_scan(_scalar_inputs([dt, dt], [b1 / dt, b2 / dt]))
    assert_close(as64(h).reshape(-1), [gold["composed"][1]], torch.float32, "composed b")


def test_closed_form_on_gpu():
    L, d = 5000, 0.01
    y, h = gpu_scan(_scalar_inputs(np.full(L, d), np.ones(L)))
    t = np.arange(L)
    want = d * (-np.expm1((t + 1) * -d)) / (-math.expm1(-d))
    assert_close(as64(y).reshape(-1), want, torch.float32, "closed form")


# -- properties of the kernel -------------------------------------------------
def test_causality_bitwise():
    w = BASE.scaled(io="bf16", seqlen=300)
    inp = make_scan_inputs(w, seed=21)
    y0, _ = gpu_scan(inp)
    t0 = 170
    pert = dict(inp)
    for k in ("u", "delta", "z"):
        t = inp[k].clone()
        t[..., t0:] = t[..., t0:] * -3.0 + 1.0
        pert[k] = t
    B = inp["B"].clone()
    B[:, t0:] += 1.0
    pert["B"] = B
    y1, _ = gpu_scan(pert)
    assert torch.equal(y0[..., :t0], y1[..., :t0]), "outputs before t0 must not change"
    assert not torch.equal(y0[..., t0:], y1[..., t0:])


def test_deterministic():
    inp = make_scan_inputs(BASE.scaled(io="bf16", seqlen=500), seed=4)
    y0, h0 = gpu_scan(inp)
    y1, h1 = gpu_scan(inp)
    assert torch.equal(y0, y1) and torch.equal(h0, h1)


# -- the full-size workloads --------------------------------------------------
@pytest.mark.parametrize("name", ["m130", "m2p8"])
def test_layer_workloads_full(name):
    check_full(WORKLOADS[name])


def test_dna_workload_sampled_channels():
    w = WORKLOADS["dna"]
    inp = make_scan_inputs(w)
    y, h = gpu_scan(inp)
    chans = sample_channels(w.batch, w.dim, 64)   # includes d = 0 and d = D - 1
    assert len(chans) == 64 and chans[0] == 0 and chans[-1] == w.dim - 1
    y_ref, h_ref = oracle_scan(inp, channels=chans)
    yv = as64(y.reshape(-1, w.seqlen)[torch.from_numpy(chans).cuda()])
    hv = as64(h.reshape(-1, w.dstate)[torch.from_numpy(chans).cuda()])
    assert_close(yv, y_ref, torch.float32, "dna y")
    assert_close(hv, h_ref, torch.float32, "dna last_state")


# -- the persistent schedule: a channel group's tokens split between two CTAs --
SPLIT = Workload("split", 3, 130, 16, 1000, "bf16", bias_range=(-4.0, -2.0),
                 a_kind="neg_exp_uniform", gate=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [4, 16])
@pytest.mark.parametrize("frac", [1.0, 1.3, 2.5, 7.0])
def test_split_groups_match_oracle(io, N, frac):
    """chunk caps the tokens one CTA scans; ranges that end inside a channel
    group hand the state over to the next CTA through the workspace."""
    w = SPLIT.scaled(io=io, dstate=N)
    inp = make_scan_inputs(w, seed=3)
    y, h = gpu_scan(inp, chunk=int(w.seqlen * frac))
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")


def test_schedule_is_bitwise_invariant():
    """Every channel's arithmetic is the same whichever CTA scans which tokens."""
    w = SPLIT.scaled(io="bf16", seqlen=777)
    inp = make_scan_inputs(w, seed=8)
    y0, h0 = gpu_scan(inp)
    for chunk in (777, 900, 1500, 2333, 5000):
        y1, h1 = gpu_scan(inp, chunk=chunk)
        assert torch.equal(y0, y1) and torch.equal(h0, h1), chunk


def test_workspace_status_word():
    """After the work finishes the workspace's first int32 reads SSM_OK."""
    import selective_state_space_116_b300 as ssm
    from parity import to_cuda
    w = SPLIT.scaled(io="f32")
    g = to_cuda(make_scan_inputs(w, seed=1))
    nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, torch.float32)
    ws = torch.full((nbytes,), 0x55, dtype=torch.uint8, device="cuda")   # stale contents
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                     delta_bias=g["delta_bias"], delta_softplus=True, workspace=ws,
                     chunk=2 * w.seqlen)
    torch.cuda.synchronize()
    assert ws[:4].view(torch.int32).item() == 0


def test_default_schedule_splits_large_problem():
    """More channel groups than resident CTAs: the default schedule splits
    groups between CTAs (8 x 3840 channels, N = 16 -> 480 groups)."""
    w = Workload("wide", 8, 3840, 16, 200, "bf16", bias_range=(-4.0, -2.0),
                 a_kind="neg_index", gate=True)
    inp = make_scan_inputs(w, seed=2)
    y, h = gpu_scan(inp)
    chans = sample_channels(w.batch, w.dim, 256)
    y_ref, h_ref = oracle_scan(inp, channels=chans)
    idx = torch.from_numpy(chans).cuda()
    assert_close(as64(y.reshape(-1, w.seqlen)[idx]), y_ref, torch.bfloat16, "y")
    assert_close(as64(h.reshape(-1, w.dstate)[idx]), h_ref, torch.bfloat16, "last_state")


# -- bf16 I/O, N = 16: many channels per group, ragged group and token counts --
TC = Workload("bf16n16", 2, 200, 16, 256, "bf16", bias_range=(-4.0, -2.0),
              a_kind="neg_exp_uniform", gate=True)


@pytest.mark.parametrize("L", [8, 16, 40, 256, 808])
@pytest.mark.parametrize("dim", [1, 127, 128, 129, 300])
def test_bf16_n16_shapes(L, dim):
    check_full(TC.scaled(seqlen=L, dim=dim, batch=1 if dim > 128 else 3), seed=L * 7 + dim)


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("softplus", [False, True])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("skip", [False, True])
def test_bf16_n16_options(gate, softplus, bias, skip):
    w = TC.scaled(gate=gate, softplus=softplus, skip=skip,
                  bias_range=(-4.0, -2.0) if bias else None)
    inp = make_scan_inputs(w, seed=13)
    if not softplus:
        inp["delta"] = (inp["delta"].float().abs() * 0.1).to(torch.bfloat16)
        if inp["delta_bias"] is not None:
            inp["delta_bias"] = inp["delta_bias"].abs() * 0.01
    y, h = gpu_scan(inp)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.bfloat16, "y")
    assert_close(as64(h), h_ref, torch.bfloat16, "last_state")


@pytest.mark.parametrize("frac", [1.0, 1.4, 3.0])
def test_bf16_n16_split_groups(frac):
    """Channel groups of 128 split between CTAs (chunk caps the tokens per CTA)."""
    w = TC.scaled(batch=3, dim=300, seqlen=800)
    inp = make_scan_inputs(w, seed=17)
    y, h = gpu_scan(inp, chunk=int(frac * w.seqlen))
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.bfloat16, "y")
    assert_close(as64(h), h_ref, torch.bfloat16, "last_state")


def test_bf16_n16_schedule_bitwise_invariant():
    w = TC.scaled(batch=2, dim=256, seqlen=512)
    inp = make_scan_inputs(w, seed=19)
    y0, h0 = gpu_scan(inp)
    for chunk in (512, 700, 1100, 2048):
        y1, h1 = gpu_scan(inp, chunk=chunk)
        assert torch.equal(y0, y1) and torch.equal(h0, h1), chunk


def test_bf16_n16_causality_bitwise():
    w = TC.scaled(seqlen=320)
    inp = make_scan_inputs(w, seed=23)
    y0, _ = gpu_scan(inp)
    t0 = 168
    pert = dict(inp)
    for k in ("u", "delta", "z"):
        t = inp[k].clone()
        t[..., t0:] = t[..., t0:] * -3.0 + 1.0
        pert[k] = t
    B = inp["B"].clone()
    B[:, t0:] += 1.0
    pert["B"] = B
    y1, _ = gpu_scan(pert)
    assert torch.equal(y0[..., :t0], y1[..., :t0])
    assert not torch.equal(y0[..., t0:], y1[..., t0:])


# -- the chunked (L-parallel) schedule -----------------------------------------
CHUNKED = Workload("chunked", 2, 70, 16, 1000, "f32", bias_range=(-4.0, -2.0),
                   a_kind="neg_exp_uniform", gate=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 4, 16])
@pytest.mark.parametrize("chunk", [32, 96, 300])
def test_chunked_matches_oracle(io, N, chunk):
    """chunk < L: the chunks' maps are found in parallel (each chunk walked
    back from its end), composed into carry-ins, and the chunks scanned from
    those."""
    w = CHUNKED.scaled(io=io, dstate=N)
    inp = make_scan_inputs(w, seed=N + chunk)
    y, h = gpu_scan(inp, chunk=chunk)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, w.torch_io, "y")
    assert_close(as64(h), h_ref, w.torch_io, "last_state")


@pytest.mark.parametrize("gate", [False, True])
@pytest.mark.parametrize("softplus", [False, True])
@pytest.mark.parametrize("skip", [False, True])
def test_chunked_options(gate, softplus, skip):
    w = CHUNKED.scaled(gate=gate, softplus=softplus, skip=skip, seqlen=777)
    inp = make_scan_inputs(w, seed=31)
    if not softplus:
        inp["delta"] = inp["delta"].abs() * 0.1
        inp["delta_bias"] = inp["delta_bias"].abs() * 0.01
    y, h = gpu_scan(inp, chunk=64)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")


@pytest.mark.parametrize("decay", ["zero_and_slow", "fast"])
def test_chunked_aggregate_walk(decay):
    """The chunked schedule's aggregate pass walks each chunk backwards from
    its end and stops once every decay product is below 2^-40.  zero_and_slow:
    states with A = 0 and A = -1e-4 (n + 1) never get there, so every chunk is
    walked to its start; fast: A = -20 makes the products negligible within
    the first tile, so the walk stops with the next tile's copy in flight."""
    w = CHUNKED.scaled(seqlen=1000)
    inp = make_scan_inputs(w, seed=41)
    A = inp["A"].clone()
    if decay == "zero_and_slow":
        A[:, ::3] = 0.0
        slow = -1e-4 * torch.arange(1, w.dstate + 1, dtype=torch.float32)
        A[1::2, 1::3] = slow[1::3]
    else:
        A[:] = -20.0
    inp["A"] = A
    for chunk in (64, 256):
        y, h = gpu_scan(inp, chunk=chunk)
        y_ref, h_ref = oracle_scan(inp)
        assert_close(as64(y), y_ref, torch.float32, f"y, chunk {chunk}")
        assert_close(as64(h), h_ref, torch.float32, f"last_state, chunk {chunk}")


def test_chunked_by_default_for_long_sequences():
    """Few channels, long sequence: the default schedule takes the chunked path
    (128 channels, L = 20000, DNA-like one-hot input)."""
    w = WORKLOADS["dna"].scaled(dim=128, seqlen=20000)
    inp = make_scan_inputs(w, seed=3)
    y, h = gpu_scan(inp)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, torch.float32, "y")
    assert_close(as64(h), h_ref, torch.float32, "last_state")
    y1, h1 = gpu_scan(inp, chunk=w.seqlen)   # one CTA range per group: no chunks
    assert_close(as64(y1), y_ref, torch.float32, "y (unchunked)")
