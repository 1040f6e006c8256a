"""B300-native selective scan (Mamba's selective state-space recurrence).

Python face of ``libssm_scan.so``: the functions here check and marshal
torch tensors into raw pointers and call the C ABI of include/ssm_scan.h
with the same names.  Every step of the scan runs in the library's CUDA
kernels; PyTorch only supplies device memory and the current stream.

Host (CPU) tensors are accepted as well: they go to ssm_scan_fwd_host, which
copies them to the current CUDA device slice by slice, overlapping the copies
with the scans on the current stream, and copies the outputs back into host
tensors (pinned when the inputs were pinned).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import SSMError, ssm_dims

__all__ = ["ssm_scan_fwd", "scan_status", "ssm_scan_bwd", "selective_scan", "ssm_state_step",
           "ssm_scan_fwd_workspace_size", "ssm_scan_bwd_workspace_size", "SSMError",
           "library_path", "version"]

_IO = {torch.float32: _lib.SSM_IO_F32, torch.bfloat16: _lib.SSM_IO_BF16}


def library_path() -> str:
    return _lib.LIBRARY


def version() -> int:
    return _lib.load().ssm_version()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(t, name, shape, dtype, device, optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _host_like(t, pinned):
    return torch.empty(t.shape, dtype=t.dtype, pin_memory=pinned)


def _dims(batch, dim, dstate, seqlen, io, chunk=0):
    return ssm_dims(int(batch), int(dim), int(dstate), int(seqlen), int(io), int(chunk))


def ssm_scan_fwd_workspace_size(batch, dim, dstate, seqlen, dtype=torch.bfloat16, chunk=0) -> int:
    """Bytes of device workspace one scan of these sizes needs."""
    out = ctypes.c_size_t(0)
    d = _dims(batch, dim, dstate, seqlen, _IO[dtype], chunk)
    rc = _lib.load().ssm_scan_fwd_workspace_size(ctypes.byref(d), ctypes.byref(out))
    if rc != 0:
        raise SSMError(rc, "ssm_scan_fwd_workspace_size")
    return int(out.value)


def ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, dtype=torch.bfloat16, chunk=0) -> int:
    """Bytes of device workspace one backward scan of these sizes needs
    (more than the checkpoints alone when the sequence is cut into chunks)."""
    out = ctypes.c_size_t(0)
    d = _dims(batch, dim, dstate, seqlen, _IO[dtype], chunk)
    rc = _lib.load().ssm_scan_bwd_workspace_size(ctypes.byref(d), ctypes.byref(out))
    if rc != 0:
        raise SSMError(rc, "ssm_scan_bwd_workspace_size")
    return int(out.value)


def _scan_fwd_host(u, delta, A, B, C, D, z, delta_bias, delta_softplus, return_last_state,
                   y, last_state, chunk):
    """Host tensors: ssm_scan_fwd_host of the library (copies in, scans and
    copies out overlapped slice by slice) on the current CUDA device and
    stream; returns once the outputs are in the host tensors."""
    cpu = torch.device("cpu")
    if u.dim() != 3 or A.dim() != 2:
        raise ValueError("u must be (batch, dim, L) and A (dim, N)")
    batch, dim, L = u.shape
    N = A.shape[1]
    io = u.dtype
    if io not in _IO:
        raise TypeError(f"unsupported I/O dtype {io}; use float32 or bfloat16")
    _check(u, "u", (batch, dim, L), io, cpu)
    _check(delta, "delta", (batch, dim, L), io, cpu)
    _check(A, "A", (dim, N), torch.float32, cpu)
    _check(B, "B", (batch, L, N), io, cpu)
    _check(C, "C", (batch, L, N), io, cpu)
    _check(D, "D", (dim,), torch.float32, cpu, optional=True)
    _check(z, "z", (batch, dim, L), io, cpu, optional=True)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, cpu, optional=True)
    pinned = u.is_pinned()
    if y is None:
        y = _host_like(u, pinned)
    _check(y, "y", (batch, dim, L), io, cpu)
    if return_last_state and last_state is None:
        last_state = torch.empty((batch, dim, N), dtype=torch.float32, pin_memory=pinned)
    if last_state is not None:
        _check(last_state, "last_state", (batch, dim, N), torch.float32, cpu)
    dev = torch.device("cuda", torch.cuda.current_device())
    st = torch.cuda.current_stream(dev)
    d = _dims(batch, dim, N, L, _IO[io], chunk)
    rc = _lib.load().ssm_scan_fwd_host(
        ctypes.byref(d), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), 1 if delta_softplus else 0, _ptr(y), _ptr(last_state), st.cuda_stream)
    if rc != 0:
        raise SSMError(rc, "ssm_scan_fwd_host")
    st.synchronize()
    return y, last_state


def ssm_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                 return_last_state=True, y=None, last_state=None, workspace=None, chunk=0,
                 input_term="delta_b", h0=None, conv_weight=None, conv_bias=None,
                 conv_state=None, u_out=None, check=False, wait_limit=0,
                 _test_skip_handoff=False):
    """Forward selective scan.

    u, delta, z: (batch, dim, L); B, C: (batch, L, N), all fp32 or all bf16.
    A: (dim, N) fp32; D, delta_bias: (dim,) fp32 or None.
    Returns (y, last_state); last_state is None unless return_last_state.
    ``y``/``last_state``/``workspace`` may be passed preallocated.

    Options (CUDA tensors; they route the call to ssm_scan_fwd_ex):
    ``input_term``: "delta_b" (Delta B u) or "zoh" ((exp(Delta A) - 1)/A B u);
    ``h0``: (batch, dim, N) fp32 initial state (may be ``last_state`` itself);
    ``conv_weight``: (dim, K) fp32, K <= 4 -- then ``u`` is the input x of the
    fused short convolution u' = silu(conv(x) + conv_bias) and the scan runs
    on u'; ``conv_bias``: (dim,) fp32; ``conv_state``: (batch, dim, K - 1)
    inputs before token 0; ``u_out``: (batch, dim, L) tensor to receive u';
    ``wait_limit``: polls of a bounded hand-over wait (0: about a second).

    ``check``: wait for the scan and raise SSMError if the device reported a
    failure (a bounded wait that gave up: the affected outputs are NaN; a
    failed bounds check of a debug build).  Without it the call returns as
    soon as the work is enqueued; ``scan_status(workspace)`` reads the same
    outcome later.  ``_test_skip_handoff`` is a test hook (see
    ssm_scan_opts.test_skip_handoff).
    """
    opts = (input_term != "delta_b" or h0 is not None or conv_weight is not None or
            wait_limit != 0 or _test_skip_handoff)
    if u.device.type == "cpu":
        if opts:
            raise ValueError("scan options take CUDA tensors")
        return _scan_fwd_host(u, delta, A, B, C, D, z, delta_bias, delta_softplus,
                              return_last_state, y, last_state, chunk)

    device = u.device
    if device.type != "cuda":
        raise ValueError("ssm_scan_fwd needs CUDA (or host) tensors")
    if u.dim() != 3 or A.dim() != 2:
        raise ValueError("u must be (batch, dim, L) and A (dim, N)")
    batch, dim, L = u.shape
    N = A.shape[1]
    io = u.dtype
    if io not in _IO:
        raise TypeError(f"unsupported I/O dtype {io}; use float32 or bfloat16")
    _check(u, "u", (batch, dim, L), io, device)
    _check(delta, "delta", (batch, dim, L), io, device)
    _check(A, "A", (dim, N), torch.float32, device)
    _check(B, "B", (batch, L, N), io, device)
    _check(C, "C", (batch, L, N), io, device)
    _check(D, "D", (dim,), torch.float32, device, optional=True)
    _check(z, "z", (batch, dim, L), io, device, optional=True)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, device, optional=True)
    if y is None:
        y = torch.empty((batch, dim, L), dtype=io, device=device)
    _check(y, "y", (batch, dim, L), io, device)
    if return_last_state and last_state is None:
        last_state = torch.empty((batch, dim, N), dtype=torch.float32, device=device)
    if last_state is not None:
        _check(last_state, "last_state", (batch, dim, N), torch.float32, device)
    d = _dims(batch, dim, N, L, _IO[io], chunk)
    lib = _lib.load()
    need = ctypes.c_size_t(0)
    rc = lib.ssm_scan_fwd_workspace_size(ctypes.byref(d), ctypes.byref(need))
    if rc != 0:
        raise SSMError(rc, "ssm_scan_fwd_workspace_size")
    if need.value and workspace is None:
        workspace = torch.empty(int(need.value), dtype=torch.uint8, device=device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(delta_softplus)), _ptr(y), _ptr(last_state), _ptr(workspace), ws_bytes,
            _stream(device))
    if not opts:
        rc = lib.ssm_scan_fwd(ctypes.byref(d), *args)
        if rc != 0:
            raise SSMError(rc, "ssm_scan_fwd")
        if check:
            scan_status(workspace, raise_on_error=True)
        return y, (last_state if return_last_state else None)
    if input_term not in ("delta_b", "zoh"):
        raise ValueError(f"input_term must be 'delta_b' or 'zoh', not {input_term!r}")
    o = _lib.ssm_scan_opts()
    o.input_term = _lib.SSM_INPUT_ZOH if input_term == "zoh" else _lib.SSM_INPUT_DELTA_B
    _check(h0, "h0", (batch, dim, N), torch.float32, device, optional=True)
    o.h0 = _ptr(h0)
    if conv_weight is not None:
        if conv_weight.dim() != 2:
            raise ValueError("conv_weight must be (dim, K)")
        K = conv_weight.shape[1]
        _check(conv_weight, "conv_weight", (dim, K), torch.float32, device)
        _check(conv_bias, "conv_bias", (dim,), torch.float32, device, optional=True)
        _check(conv_state, "conv_state", (batch, dim, K - 1), io, device, optional=True)
        _check(u_out, "u_out", (batch, dim, L), io, device, optional=True)
        o.conv_width = K
        o.conv_weight, o.conv_bias = _ptr(conv_weight), _ptr(conv_bias)
        o.conv_state, o.u_out = _ptr(conv_state), _ptr(u_out)
    elif conv_bias is not None or conv_state is not None or u_out is not None:
        raise ValueError("conv_bias, conv_state and u_out need conv_weight")
    o.wait_limit = int(wait_limit)
    o.test_skip_handoff = 1 if _test_skip_handoff else 0
    rc = lib.ssm_scan_fwd_ex(ctypes.byref(d), ctypes.byref(o), *args)
    if rc != 0:
        raise SSMError(rc, "ssm_scan_fwd_ex")
    if check:
        scan_status(workspace, raise_on_error=True)
    return y, (last_state if return_last_state else None)


def scan_status(workspace, raise_on_error=False) -> int:
    """The device-side outcome of the last scan that used ``workspace`` (a
    CUDA uint8 tensor, or None for a scan that needed none): waits for the
    current stream, then returns 0 or a negative status (SSM_ERR_TIMEOUT,
    SSM_ERR_DEVICE), raising SSMError instead when ``raise_on_error``."""
    lib = _lib.load()
    if workspace is None:
        rc = 0
    else:
        rc = lib.ssm_scan_fwd_status(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(workspace.device))
    if rc != 0 and raise_on_error:
        raise SSMError(rc, "scan on the device")
    return rc


def ssm_state_step(state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                   delta_softplus=False, y=None):
    """One generation step: updates ``state`` (batch, dim, N) fp32 in place
    and returns y (batch, dim).  x, delta, z: (batch, dim); B, C: (batch, N)."""
    device = state.device
    if device.type != "cuda":
        raise ValueError("ssm_state_step needs CUDA tensors")
    if state.dim() != 3:
        raise ValueError("state must be (batch, dim, N)")
    batch, dim, N = state.shape
    io = x.dtype
    if io not in _IO:
        raise TypeError(f"unsupported I/O dtype {io}; use float32 or bfloat16")
    _check(state, "state", (batch, dim, N), torch.float32, device)
    _check(x, "x", (batch, dim), io, device)
    _check(delta, "delta", (batch, dim), io, device)
    _check(A, "A", (dim, N), torch.float32, device)
    _check(B, "B", (batch, N), io, device)
    _check(C, "C", (batch, N), io, device)
    _check(D, "D", (dim,), torch.float32, device, optional=True)
    _check(z, "z", (batch, dim), io, device, optional=True)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, device, optional=True)
    if y is None:
        y = torch.empty((batch, dim), dtype=io, device=device)
    _check(y, "y", (batch, dim), io, device)
    d = _dims(batch, dim, N, 1, _IO[io])
    rc = _lib.load().ssm_state_step(ctypes.byref(d), _ptr(state), _ptr(x), _ptr(delta), _ptr(A),
                                    _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
                                    int(bool(delta_softplus)), _ptr(y), _stream(device))
    if rc != 0:
        raise SSMError(rc, "ssm_state_step")
    return y


def ssm_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=False,
                 dlast_state=None, return_dh0=False, workspace=None, h0=None,
                 input_term="delta_b", chunk=0, grad_dtype=torch.float32):
    """Backward selective scan (CUDA tensors): the gradients of a loss with
    dLoss/dy = ``dy`` (and dLoss/dlast_state = ``dlast_state``) with respect
    to the inputs of ``ssm_scan_fwd`` run from the initial state ``h0``
    ((batch, dim, N) fp32, or None for zero) with the input term
    ``input_term`` ("delta_b" or "zoh", as for ``ssm_scan_fwd``).
    The forward states are recomputed inside the kernel.  ``chunk``: 0 for
    the library's schedule (long sequences over few channels are cut into
    chunks run side by side), else chunks of about that many tokens
    (ssm_dims.chunk).  ``grad_dtype``: float32, or the I/O dtype: the dtype
    of ``dy`` and of du, ddelta and dz (written as the fp32 values rounded
    once).
    Returns a dict of
    tensors: du, ddelta (gradient of the raw delta), dz (None without
    z), dA, dB, dC, dD (None without D), ddelta_bias (None without
    delta_bias) and dh0 (None unless ``return_dh0``).
    """
    device = u.device
    if device.type != "cuda":
        raise ValueError("ssm_scan_bwd needs CUDA tensors")
    batch, dim, L = u.shape
    N = A.shape[1]
    io = u.dtype
    if io not in _IO:
        raise TypeError(f"unsupported I/O dtype {io}; use float32 or bfloat16")
    _check(u, "u", (batch, dim, L), io, device)
    _check(delta, "delta", (batch, dim, L), io, device)
    _check(A, "A", (dim, N), torch.float32, device)
    _check(B, "B", (batch, L, N), io, device)
    _check(C, "C", (batch, L, N), io, device)
    _check(D, "D", (dim,), torch.float32, device, optional=True)
    _check(z, "z", (batch, dim, L), io, device, optional=True)
    _check(delta_bias, "delta_bias", (dim,), torch.float32, device, optional=True)
    if grad_dtype not in (torch.float32, io):
        raise TypeError(f"grad_dtype must be float32 or the I/O dtype {io}, not {grad_dtype}")
    _check(dy, "dy", (batch, dim, L), grad_dtype, device)
    _check(dlast_state, "dlast_state", (batch, dim, N), torch.float32, device, optional=True)
    _check(h0, "h0", (batch, dim, N), torch.float32, device, optional=True)
    if input_term not in ("delta_b", "zoh"):
        raise ValueError(f"input_term must be 'delta_b' or 'zoh', not {input_term!r}")
    term = _lib.SSM_INPUT_ZOH if input_term == "zoh" else _lib.SSM_INPUT_DELTA_B
    f32 = dict(dtype=torch.float32, device=device)
    gt = dict(dtype=grad_dtype, device=device)
    g = {"du": torch.empty((batch, dim, L), **gt), "ddelta": torch.empty((batch, dim, L), **gt),
         "dz": torch.empty((batch, dim, L), **gt) if z is not None else None,
         "dA": torch.empty((dim, N), **f32), "dB": torch.empty((batch, L, N), **f32),
         "dC": torch.empty((batch, L, N), **f32),
         "dD": torch.empty((dim,), **f32) if D is not None else None,
         "ddelta_bias": torch.empty((dim,), **f32) if delta_bias is not None else None,
         "dh0": torch.empty((batch, dim, N), **f32) if return_dh0 else None}
    lib = _lib.load()
    d = _dims(batch, dim, N, L, _IO[io], chunk)
    need = ctypes.c_size_t(0)
    rc = lib.ssm_scan_bwd_workspace_size(ctypes.byref(d), ctypes.byref(need))
    if rc != 0:
        raise SSMError(rc, "ssm_scan_bwd_workspace_size")
    if workspace is None and need.value > 0:
        workspace = torch.empty(need.value, dtype=torch.uint8, device=device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.ssm_scan_bwd_ex(ctypes.byref(d), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                             _ptr(D), _ptr(z), _ptr(delta_bias), 1 if delta_softplus else 0,
                             _ptr(dy), _ptr(dlast_state), _ptr(h0), term, _IO[grad_dtype],
                             _ptr(g["du"]),
                             _ptr(g["ddelta"]), _ptr(g["dz"]), _ptr(g["dA"]), _ptr(g["dB"]),
                             _ptr(g["dC"]), _ptr(g["dD"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
                             _ptr(workspace), ws_bytes, _stream(device))
    if rc != 0:
        raise SSMError(rc, "ssm_scan_bwd_ex")
    return g


class _SelectiveScan(torch.autograd.Function):
    """Forward through ssm_scan_fwd, backward through ssm_scan_bwd (which
    recomputes the forward states; nothing but the inputs is saved)."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, input_term):
        y, last = ssm_scan_fwd(u, delta, A, B, C, D=D, z=z, delta_bias=delta_bias,
                               delta_softplus=delta_softplus, return_last_state=True, h0=h0,
                               input_term=input_term)
        ctx.save_for_backward(u, delta, A, B, C, D, z, delta_bias, h0)
        ctx.delta_softplus = delta_softplus
        ctx.input_term = input_term
        return y, last

    @staticmethod
    def backward(ctx, dy, dlast):
        u, delta, A, B, C, D, z, delta_bias, h0 = ctx.saved_tensors
        dy = torch.zeros_like(u) if dy is None else dy.to(u.dtype).contiguous()
        dlast = None if dlast is None else dlast.float().contiguous()
        want_dh0 = h0 is not None and ctx.needs_input_grad[9]
        # dy goes in, and du, ddelta, dz come out, in the inputs' dtype (u,
        # delta, z and y share it)
        g = ssm_scan_bwd(u, delta, A, B, C, dy, D=D, z=z, delta_bias=delta_bias,
                         delta_softplus=ctx.delta_softplus, dlast_state=dlast, h0=h0,
                         return_dh0=want_dh0, input_term=ctx.input_term, grad_dtype=u.dtype)
        cast = lambda t, like: None if t is None else t.to(like.dtype)
        return (cast(g["du"], u), cast(g["ddelta"], delta), g["dA"], cast(g["dB"], B),
                cast(g["dC"], C), g["dD"] if D is not None else None,
                cast(g["dz"], z) if z is not None else None,
                g["ddelta_bias"] if delta_bias is not None else None, None,
                g["dh0"] if want_dh0 else None, None)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                   h0=None, input_term="delta_b"):
    """Differentiable forward scan on CUDA tensors: returns (y, last_state)
    and, under autograd, gradients for every tensor input from the library's
    backward kernel, h0 (the initial state, (batch, dim, N) fp32, or None for
    zero) included.  ``input_term`` is "delta_b" or "zoh", as for
    ``ssm_scan_fwd``.  Gradients are computed in fp32 and returned in each
    input's dtype."""
    if input_term not in ("delta_b", "zoh"):
        raise ValueError(f"input_term must be 'delta_b' or 'zoh', not {input_term!r}")
    return _SelectiveScan.apply(u, delta, A, B, C, D, z, delta_bias, bool(delta_softplus), h0,
                                input_term)
