"""Single-token state update (generation) parity: against the fp64 oracle's
step, and against the CUDA scan over the same token stream."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_116_b300 as ssm
from parity import as64, assert_close, gpu_scan, oracle_scan, to_cuda
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
