"""ssm_scan_fwd_host: the scan from host buffers, with the copies overlapped
slice by slice.  Each slice is an independent scan (a batch row, or a range
of its channels), so the outputs must equal those of the device entry point
bit for bit, and match the fp64 oracle within the stated tolerances."""
import numpy as np
import pytest
import torch

import selective_state_space_116_b300 as ssm
from parity import as64, assert_close, gpu_scan, oracle_scan
from selective_state_space_116_b300.workloads import WORKLOADS, make_scan_inputs

pytestmark = pytest.mark.gpu


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality (NaN payloads included)."""
    a, b = a.contiguous(), b.contiguous()
    iv = torch.int16 if a.element_size() == 2 else torch.int32
    return a.shape == b.shape and a.dtype == b.dtype and torch.equal(a.view(iv), b.view(iv))


def host_scan(inp, pinned, return_last_state=True):
    h = {k: (v.pin_memory() if (pinned and isinstance(v, torch.Tensor)) else v) for k, v in inp.items()}
    return ssm.ssm_scan_fwd(h["u"], h["delta"], h["A"], h["B"], h["C"], D=h["D"], z=h["z"],
                            delta_bias=h["delta_bias"], delta_softplus=h["delta_softplus"],
                            return_last_state=return_last_state)


# (batch, dim, L): 17 batch rows (one slice a row), rows cut into channel
# ranges (with a short last range)
SHAPES = [(17, 24, 100), (4, 96, 300), (1, 300, 257), (2, 130, 64), (5, 64, 33)]


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("pinned", [True, False])
def test_host_matches_device_bitwise(io, shape, pinned):
    b, d, L = shape
    w = WORKLOADS["m130"].scaled(batch=b, dim=d, seqlen=L, last_state=True)
    if io == "f32":
        w = w.scaled(io="f32")
    inp = make_scan_inputs(w, seed=3)
    y_d, h_d = gpu_scan(inp)
    y_h, h_h = host_scan(inp, pinned)
    assert y_h.device.type == "cpu" and h_h.device.type == "cpu"
    assert y_h.is_pinned() == pinned
    assert same_bits(y_h, y_d.cpu()), "y differs from the device path"
    assert same_bits(h_h, h_d.cpu()), "last_state differs from the device path"


@pytest.mark.parametrize("N", [1, 4, 16])
def test_host_matches_oracle(N):
    w = WORKLOADS["m130"].scaled(batch=3, dim=70, seqlen=129, dstate=N, last_state=True)
    inp = make_scan_inputs(w, seed=5)
    y, h = host_scan(inp, pinned=True)
    y_ref, h_ref = oracle_scan(inp)
    assert_close(as64(y), y_ref, w.torch_io, "host y")
    assert_close(as64(h), h_ref, w.torch_io, "host last_state")


def test_host_options_and_empty():
    w = WORKLOADS["m130"].scaled(batch=2, dim=40, seqlen=48, last_state=True)
    inp = make_scan_inputs(w, seed=7)
    # no gate, skip, bias or softplus: Delta = delta itself, kept positive
    inp = dict(inp, z=None, D=None, delta_bias=None, delta_softplus=False, delta=inp["delta"].abs())
    y_d, _ = gpu_scan(inp, return_last_state=False)
    y_h, h_h = host_scan(inp, pinned=True, return_last_state=False)
    assert h_h is None
    assert torch.isfinite(y_h.float()).all()
    assert same_bits(y_h, y_d.cpu())
    # L = 0: empty outputs, zero last state
    w0 = w.scaled(seqlen=0)
    inp0 = make_scan_inputs(w0, seed=1)
    y0, h0 = host_scan(inp0, pinned=False)
    assert y0.shape == (2, 40, 0)
    assert torch.count_nonzero(h0) == 0


def test_host_full_layer_sampled():
    """The Mamba-2.8B layer shape from pinned buffers: equal to the device path."""
    w = WORKLOADS["m2p8"]
    inp = make_scan_inputs(w, seed=0)
    y_d, h_d = gpu_scan(inp)
    y_h, h_h = host_scan(inp, pinned=True)
    assert same_bits(y_h, y_d.cpu())
    assert same_bits(h_h, h_d.cpu())
