"""Failure detection on the GPU without a fault: the bounded hand-over wait
of the persistent schedule runs out (a test hook withholds the flags that
publish the hand-overs), the kernel gives up after a short limit, writes NaN
to what it could not compute and leaves SSM_ERR_TIMEOUT for the status
query; the device stays usable.  Also: guard bands around every output stay
untouched, and the allocation-free entry point's status is readable."""
import ctypes

import numpy as np
import pytest
import torch

import selective_state_space_116_b300 as ssm
from parity import as64, assert_close, gpu_scan, oracle_scan, to_cuda
from selective_state_space_116_b300 import _lib
from selective_state_space_116_b300.workloads import Workload, make_scan_inputs

pytestmark = pytest.mark.gpu

# 3 x 130 channels, N = 16: with chunk = 1.3 L the persistent schedule splits
# channel groups between CTAs, which hand the state over through the workspace
SPLIT = Workload("split", 3, 130, 16, 1000, "f32", bias_range=(-4.0, -2.0),
                 a_kind="neg_exp_uniform", gate=True)


def _scan(g, w, ws, **kw):
    return ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                            delta_bias=g["delta_bias"], delta_softplus=True, workspace=ws,
                            chunk=int(1.3 * w.seqlen), **kw)


def test_withheld_handover_times_out_and_is_reported():
    w = SPLIT
    inp = make_scan_inputs(w, seed=70)
    g = to_cuda(inp)
    nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, torch.float32,
                                             chunk=int(1.3 * w.seqlen))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    # 2000 polls ~ 0.5 ms: the waits give up quickly
    y, h = _scan(g, w, ws, wait_limit=2000, _test_skip_handoff=True)
    assert ssm.scan_status(ws) == _lib.SSM_ERR_TIMEOUT
    with pytest.raises(ssm.SSMError) as err:
        _scan(g, w, ws, wait_limit=2000, _test_skip_handoff=True, check=True)
    assert err.value.status == _lib.SSM_ERR_TIMEOUT
    # the channels whose tail could not be computed are NaN from the hand-over
    # point on; everything else equals the oracle
    y64, h64 = as64(y), as64(h)
    y_ref, h_ref = oracle_scan(inp)
    bad_y, bad_h = np.isnan(y64), np.isnan(h64).any(-1)
    assert bad_y.any() and bad_h.any()
    for b in range(w.batch):
        for d in range(w.dim):
            row = bad_y[b, d]
            if row.any():
                first = int(np.argmax(row))
                assert row[first:].all(), "NaN must run to the end of the sequence"
                assert bad_h[b, d]
    assert_close(np.where(bad_y, y_ref, y64), y_ref, torch.float32, "y outside the gap")
    ok = ~bad_h
    assert_close(h64[ok], h_ref[ok], torch.float32, "last_state outside the gap")
    # the device is still usable: the same call without the hook is correct
    y, h = _scan(g, w, ws, check=True)
    assert ssm.scan_status(ws) == _lib.SSM_OK
    assert_close(as64(y), y_ref, torch.float32, "y after the timeout")
    assert_close(as64(h), h_ref, torch.float32, "last_state after the timeout")


def test_status_of_clean_calls():
    w = SPLIT.scaled(seqlen=300)
    g = to_cuda(make_scan_inputs(w, seed=71))
    nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, torch.float32)
    ws = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")   # stale contents
    ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                     delta_bias=g["delta_bias"], delta_softplus=True, workspace=ws)
    assert ssm.scan_status(ws) == _lib.SSM_OK
    # the allocation-free entry keeps its status in its own buffer
    lib = _lib.load()
    d = _lib.ssm_dims(w.batch, w.dim, w.dstate, w.seqlen, _lib.SSM_IO_F32, 0)
    y = torch.empty_like(g["u"])
    p = lambda t: None if t is None else t.data_ptr()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.ssm_scan_fwd_noalloc(ctypes.byref(d), p(g["u"]), p(g["delta"]), p(g["A"]), p(g["B"]),
                                  p(g["C"]), p(g["D"]), p(g["z"]), p(g["delta_bias"]), 1, p(y),
                                  None, stream)
    assert rc == _lib.SSM_OK
    assert lib.ssm_scan_fwd_noalloc_status(stream) == _lib.SSM_OK


GUARD = 4096   # bytes of guard band on each side of an output


def _guarded(shape, dtype):
    """An output tensor inside a buffer with guard bands of a fixed pattern."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    t = buf[GUARD:GUARD + n].view(dtype).view(*shape)
    return buf, t


def _guards_intact(buf):
    return bool((buf[:GUARD] == 0xA5).all() and (buf[-GUARD:] == 0xA5).all())


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L,dim,N", [(1, 1, 16), (7, 65, 4), (33, 130, 16), (257, 3, 1), (1000, 64, 8)])
@pytest.mark.parametrize("conv", [False, True])
def test_outputs_stay_inside_their_buffers(io, L, dim, N, conv):
    """Guard bands before and after y, last_state and the convolution output
    are untouched by scans over ragged shapes (every schedule and path)."""
    w = SPLIT.scaled(io=io, seqlen=L, dim=dim, dstate=N, batch=2)
    inp = make_scan_inputs(w, seed=L + dim)
    g = to_cuda(inp)
    ybuf, y = _guarded((2, dim, L), w.torch_io)
    hbuf, h = _guarded((2, dim, N), torch.float32)
    ubuf, u_out = _guarded((2, dim, L), w.torch_io)
    kw = dict(conv_weight=torch.randn(dim, 4, device="cuda"), u_out=u_out) if conv else {}
    for chunk in (0, 32, int(1.5 * L)):
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                         delta_bias=g["delta_bias"], delta_softplus=True, y=y, last_state=h,
                         chunk=chunk, check=True, **kw)
        torch.cuda.synchronize()
        assert _guards_intact(ybuf) and _guards_intact(hbuf), chunk
        if conv:
            assert _guards_intact(ubuf), chunk
