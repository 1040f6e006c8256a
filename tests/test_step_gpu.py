"""Single-token state update (generation) parity: against the fp64 oracle's
step, and against the CUDA scan over the same token stream."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_116_b300 as ssm
from parity import TOL, as64, assert_close, gpu_scan, oracle_scan, to_cuda
from selective_state_space_116_b300.workloads import (WORKLOADS, make_step_inputs,
                                                      steps_as_scan)

pytestmark = pytest.mark.gpu


def gpu_steps(inp, steps, state=None, record_states=()):
    g = to_cuda(inp)
    T, batch, dim = g["x"].shape
    N = g["A"].shape[1]
    if state is None:
        state = torch.zeros(batch, dim, N, device="cuda")
    ys, states = [], {}
    for t in range(steps):
        y = ssm.ssm_state_step(state, g["x"][t], g["delta"][t], g["A"], g["B"][t], g["C"][t],
                               D=g["D"], z=None if g["z"] is None else g["z"][t],
                               delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"])
        ys.append(y.clone())
        if t + 1 in record_states:
            states[t + 1] = state.clone()
    torch.cuda.synchronize()
    return torch.stack(ys), state, states


def oracle_steps(inp, steps):
    T, batch, dim = inp["x"].shape
    N = inp["A"].shape[1]
    state = np.zeros((batch, dim, N))
    ys = []
    for t in range(steps):
        ys.append(oracle.state_step(state, inp["x"][t], inp["delta"][t], inp["A"], inp["B"][t],
                                    inp["C"][t], D=inp["D"],
                                    z=None if inp["z"] is None else inp["z"][t],
                                    delta_bias=inp["delta_bias"],
                                    delta_softplus=inp["delta_softplus"]))
    return np.stack(ys), state


SMALL = WORKLOADS["gen"].scaled(batch=3, dim=70, steps=40)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
def test_steps_match_oracle(io, N):
    w = SMALL.scaled(io=io, dstate=N, a_kind="neg_exp_uniform")
    inp = make_step_inputs(w, seed=N)
    y, state, _ = gpu_steps(inp, w.steps)
    y_ref, state_ref = oracle_steps(inp, w.steps)
    assert_close(as64(y), y_ref, w.torch_io, "step y")
    assert_close(as64(state), state_ref, w.torch_io, "step state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_match_scan(io):
    """Per-step outputs equal the scan's y_t; the state after k steps equals the
    last_state of a scan over the first k tokens."""
    w = SMALL.scaled(io=io)
    inp = make_step_inputs(w, seed=7)
    y, state, states = gpu_steps(inp, w.steps, record_states=(1, 2, 17, w.steps))
    s = steps_as_scan(inp)
    ys, hs = gpu_scan(s)
    assert_close(as64(y), as64(ys.permute(2, 0, 1)), w.torch_io, "step y vs scan y")
    for k, st in states.items():
        pre = dict(s)
        for key in ("u", "delta", "z"):
            pre[key] = None if s[key] is None else s[key][..., :k].contiguous()
        for key in ("B", "C"):
            pre[key] = s[key][:, :k].contiguous()
        _, hk = gpu_scan(pre)
        assert_close(as64(st), as64(hk), w.torch_io, f"state after {k} steps")


def test_scan_then_steps_resumes():
    """last_state is a checkpoint: scan the first k tokens, continue with steps."""
    w = SMALL.scaled(io="f32")
    inp = make_step_inputs(w, seed=9)
    s = steps_as_scan(inp)
    k = 25
    pre = {key: (None if v is None else v) for key, v in s.items()}
    for key in ("u", "delta", "z"):
        pre[key] = s[key][..., :k].contiguous()
    for key in ("B", "C"):
        pre[key] = s[key][:, :k].contiguous()
    _, hk = gpu_scan(pre)
    rest = {key: (v[k:].contiguous() if key in ("x", "delta", "z", "B", "C") and v is not None
                  else v) for key, v in inp.items()}
    y, state, _ = gpu_steps(rest, w.steps - k, state=hk.clone())
    y_ref, h_ref = oracle_scan(s)
    assert_close(as64(y), y_ref[..., k:].transpose(2, 0, 1), torch.float32, "resumed y")
    assert_close(as64(state), h_ref, torch.float32, "resumed state")


def test_generation_workload_full_size():
    """The full 128 x 5120 batch for 8 consecutive tokens against the oracle."""
    w = WORKLOADS["gen"]
    inp = make_step_inputs(w, seed=0, steps=8)
    y, state, _ = gpu_steps(inp, 8)
    y_ref, state_ref = oracle_steps(inp, 8)
    assert_close(as64(y), y_ref, torch.bfloat16, "gen y")
    assert_close(as64(state), state_ref, torch.bfloat16, "gen state")


def _close_on_gpu(got, ref, io_dtype, what):
    """assert_close's bound, evaluated on the GPU (the full generation run has
    671 M outputs per comparison)."""
    got, ref = got.double(), ref.double()
    ratio = (got - ref).abs() / (TOL[io_dtype] * (1.0 + ref.abs()))
    assert torch.isfinite(got).all(), f"{what}: non-finite output"
    worst = ratio.max().item()
    assert worst <= 1.0, f"{what}: worst scaled error {worst:.3f} of the bound"


def _prefix(s, k):
    pre = dict(s)
    for key in ("u", "delta", "z"):
        pre[key] = None if s[key] is None else s[key][..., :k].contiguous()
    for key in ("B", "C"):
        pre[key] = s[key][:, :k].contiguous()
    return pre


def test_generation_1024_steps_full_size():
    """The generation workload as configured: 128 x 5120 channels, N = 16,
    bf16 inputs, fp32 state, 1024 consecutive ssm_state_step tokens from a
    zero state.  Every step's y against the GPU scan of the same token stream;
    the state after k = 1, 2, 17, 1024 steps against the last_state of the
    GPU scan of the first k tokens; and both against the fp64 oracle on 64
    sampled channels (d = 0 and d = D - 1 of every batch row among them).
    The oracle side runs the oracle's scan over the stream, which its own
    pins tie to its single-token step."""
    w = WORKLOADS["gen"]
    steps = 1024
    K = (1, 2, 17, steps)
    inp = make_step_inputs(w, seed=0, steps=steps)
    g = to_cuda(inp)
    batch, dim, N = w.batch, w.dim, w.dstate
    state = torch.zeros(batch, dim, N, device="cuda")
    ys = torch.empty(steps, batch, dim, dtype=g["x"].dtype, device="cuda")
    states = {}
    for t in range(steps):
        ssm.ssm_state_step(state, g["x"][t], g["delta"][t], g["A"], g["B"][t], g["C"][t],
                           D=g["D"], z=g["z"][t], delta_bias=g["delta_bias"],
                           delta_softplus=g["delta_softplus"], y=ys[t])
        if t + 1 in K:
            states[t + 1] = state.clone()
    torch.cuda.synchronize()
    s = steps_as_scan(inp)
    sg = to_cuda(s)
    y_scan, h_scan = ssm.ssm_scan_fwd(sg["u"], sg["delta"], sg["A"], sg["B"], sg["C"], D=sg["D"],
                                      z=sg["z"], delta_bias=sg["delta_bias"],
                                      delta_softplus=sg["delta_softplus"])
    _close_on_gpu(ys.permute(1, 2, 0), y_scan, torch.bfloat16, "every step's y vs scan y")
    for k in K:
        if k == steps:
            hk = h_scan
        else:
            p = _prefix(sg, k)
            _, hk = ssm.ssm_scan_fwd(p["u"], p["delta"], p["A"], p["B"], p["C"], D=p["D"],
                                     z=p["z"], delta_bias=p["delta_bias"],
                                     delta_softplus=p["delta_softplus"])
        _close_on_gpu(states[k], hk, torch.bfloat16, f"state after {k} steps vs scan")
    # 64 channels: d = 0 and d = D - 1 of the first and last batch rows, the
    # rest drawn at random
    rng = np.random.default_rng(5)
    must = {0, dim - 1, (batch - 1) * dim, batch * dim - 1}
    rest = [int(c) for c in rng.choice(batch * dim, 80, replace=False) if int(c) not in must]
    chans = np.array(sorted(must | set(rest[:64 - len(must)])), dtype=np.int64)
    assert len(chans) == 64
    idx = torch.from_numpy(chans).cuda()
    y_ref, h_ref = oracle_scan(s, channels=chans)
    y_got = ys.permute(1, 2, 0).reshape(batch * dim, steps)[idx]
    assert_close(as64(y_got), y_ref, torch.bfloat16, "step y vs oracle (64 channels)")
    for k in K:
        _, hk_ref = (y_ref, h_ref) if k == steps else oracle_scan(_prefix(s, k), channels=chans)
        hk = states[k].reshape(batch * dim, N)[idx]
        assert_close(as64(hk), hk_ref, torch.bfloat16, f"state after {k} steps vs oracle")
