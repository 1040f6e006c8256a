"""The allocation-free scan, ssm_scan_fwd_noalloc, through the C ABI.

It serves callers that cannot allocate device memory when they call the scan
(for example an inference engine's plugin confined to a memory plan fixed in
advance); its scratch is a fixed buffer inside the library instead of a
caller-supplied workspace.  These tests check that two calls in a row give
the outputs of ssm_scan_fwd with a workspace, within the parity tolerance
(1e-4 (1 + |ref|) for fp32 I/O, 2e-2 (1 + |ref|) for bf16 I/O).  The file is
named to be collected last, so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import selective_state_space_116_b300 as ssm
from parity import as64, assert_close, to_cuda
from selective_state_space_116_b300 import _lib
from selective_state_space_116_b300.workloads import Workload, make_scan_inputs

pytestmark = pytest.mark.gpu

# 3 x 130 channels, N = 16, 1000 tokens; with chunk = 1.3 L the tokens of some
# channel groups are split between two CTAs, so the state is handed over
# through the scratch buffer; with chunk = 0.3 L the chunked schedule keeps
# its chunk aggregates and carries there instead.
W = Workload("noalloc", 3, 130, 16, 1000, "bf16", bias_range=(-4.0, -2.0),
             a_kind="neg_exp_uniform", gate=True)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc(g, w, chunk, y, last):
    lib = _lib.load()
    io = _lib.SSM_IO_BF16 if w.io == "bf16" else _lib.SSM_IO_F32
    d = _lib.ssm_dims(w.batch, w.dim, w.dstate, w.seqlen, io, chunk)
    rc = lib.ssm_scan_fwd_noalloc(ctypes.byref(d), _ptr(g["u"]), _ptr(g["delta"]), _ptr(g["A"]),
                                  _ptr(g["B"]), _ptr(g["C"]), _ptr(g["D"]), _ptr(g["z"]),
                                  _ptr(g["delta_bias"]), int(g["delta_softplus"]), _ptr(y),
                                  _ptr(last), torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.SSM_OK, _lib.status_string(rc)


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("frac", [0.0, 1.3, 0.3])
def test_noalloc_matches_workspace_entry(io, frac):
    w = W.scaled(io=io)
    g = to_cuda(make_scan_inputs(w, seed=5))
    chunk = int(frac * w.seqlen)
    y_ref, h_ref = ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"],
                                    z=g["z"], delta_bias=g["delta_bias"],
                                    delta_softplus=g["delta_softplus"], chunk=chunk)
    for call in range(2):   # the buffer keeps the previous call's contents
        y = torch.full_like(y_ref, float("nan"))
        last = torch.full_like(h_ref, float("nan"))
        _noalloc(g, w, chunk, y, last)
        torch.cuda.synchronize()
        assert_close(as64(y), as64(y_ref), w.torch_io, f"call {call} y")
        assert_close(as64(last), as64(h_ref), w.torch_io, f"call {call} last_state")
