"""The C ABI without a GPU: the library loads, exports every entry point that
include/*.h declares, and rejects bad arguments on the host.

Every call here fails argument validation before anything is enqueued, so the
placeholder pointer values below are never dereferenced by host or device.
"""
import ctypes
import glob
import os
import re

import pytest

from selective_state_space_116_b300 import _lib
from selective_state_space_116_b300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"SSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    declared = declared_functions()
    assert declared, "no SSM_API declarations found"
    for name in declared:
        assert hasattr(lib, name), f"{name} declared but not exported"
    assert sorted(_lib.EXPORTS) == declared


def test_version_and_status_strings(lib):
    assert lib.ssm_version() >= 100
    for code in range(0, -12, -1):
        s = _lib.status_string(code)
        assert s and s != "unknown status", code
    assert _lib.status_string(-99) == "unknown status"


# placeholder addresses: aligned, far apart, never dereferenced
P = [0x10000000 * (i + 1) for i in range(16)]


def dims(batch=2, dim=8, dstate=16, seqlen=64, io=_lib.SSM_IO_BF16, chunk=0):
    return _lib.ssm_dims(batch, dim, dstate, seqlen, io, chunk)


def scan(lib, d, u=P[0], delta=P[1], A=P[2], B=P[3], C=P[4], D=P[5], z=P[6], bias=P[7],
         y=P[8], last=P[9], ws=None, ws_bytes=0):
    return lib.ssm_scan_fwd(ctypes.byref(d) if d is not None else None, u, delta, A, B, C, D, z,
                            bias, 1, y, last, ws, ws_bytes, None)


def step(lib, d, state=P[0], x=P[1], delta=P[2], A=P[3], B=P[4], C=P[5], D=P[6], z=P[7],
         bias=P[8], y=P[9]):
    return lib.ssm_state_step(ctypes.byref(d) if d is not None else None, state, x, delta, A,
                              B, C, D, z, bias, 1, y, None)


@pytest.mark.parametrize("kw,code", [
    (dict(batch=0), _lib.SSM_ERR_BAD_DIMS),
    (dict(dim=0), _lib.SSM_ERR_BAD_DIMS),
    (dict(seqlen=-1), _lib.SSM_ERR_BAD_DIMS),
    (dict(dstate=3), _lib.SSM_ERR_UNSUPPORTED_N),
    (dict(dstate=32), _lib.SSM_ERR_UNSUPPORTED_N),
    (dict(dstate=0), _lib.SSM_ERR_BAD_DIMS),
    (dict(io=7), _lib.SSM_ERR_BAD_DTYPE),
    (dict(chunk=-64), _lib.SSM_ERR_BAD_DIMS),
    (dict(chunk=-1), _lib.SSM_ERR_BAD_DIMS),
    (dict(batch=1 << 40, dim=1 << 40), _lib.SSM_ERR_BAD_DIMS),
    (dict(batch=70000), _lib.SSM_ERR_BAD_DIMS),
])
def test_scan_rejects_bad_dims(lib, kw, code):
    assert scan(lib, dims(**kw)) == code
    out = ctypes.c_size_t(123)
    if code != _lib.SSM_OK:
        assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(dims(**kw)), ctypes.byref(out)) == code


def test_scan_null_arguments(lib):
    assert scan(lib, None) == _lib.SSM_ERR_NULL_ARG
    for name in ("u", "delta", "A", "B", "C", "y"):
        assert scan(lib, dims(), **{name: None}) == _lib.SSM_ERR_NULL_ARG, name
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(dims()), None) == _lib.SSM_ERR_NULL_ARG


def test_scan_misaligned(lib):
    assert scan(lib, dims(io=_lib.SSM_IO_BF16), u=P[0] + 1) == _lib.SSM_ERR_MISALIGNED
    assert scan(lib, dims(io=_lib.SSM_IO_F32), y=P[8] + 2) == _lib.SSM_ERR_MISALIGNED
    assert scan(lib, dims(), A=P[2] + 2) == _lib.SSM_ERR_MISALIGNED
    assert scan(lib, dims(), last=P[9] + 1) == _lib.SSM_ERR_MISALIGNED


def test_scan_aliasing(lib):
    d = dims(batch=2, dim=8, dstate=16, seqlen=64)
    assert scan(lib, d, y=P[0]) == _lib.SSM_ERR_ALIAS            # y == u
    assert scan(lib, d, y=P[0] + 64) == _lib.SSM_ERR_ALIAS       # y inside u
    assert scan(lib, d, last=P[3] + 16) == _lib.SSM_ERR_ALIAS    # last_state inside B
    assert scan(lib, d, last=P[8]) == _lib.SSM_ERR_ALIAS         # last_state == y


def test_step_errors(lib):
    assert step(lib, None) == _lib.SSM_ERR_NULL_ARG
    assert step(lib, dims(dstate=5)) == _lib.SSM_ERR_UNSUPPORTED_N
    assert step(lib, dims(io=9)) == _lib.SSM_ERR_BAD_DTYPE
    for name in ("state", "x", "delta", "A", "B", "C", "y"):
        assert step(lib, dims(), **{name: None}) == _lib.SSM_ERR_NULL_ARG, name
    assert step(lib, dims(), x=P[1] + 1) == _lib.SSM_ERR_MISALIGNED
    assert step(lib, dims(), state=P[0] + 2) == _lib.SSM_ERR_MISALIGNED
    assert step(lib, dims(), y=P[0]) == _lib.SSM_ERR_ALIAS       # y == state


def test_binding_fails_loudly_without_library(tmp_path):
    missing = os.path.join(tmp_path, "nope.so")
    saved = _lib._lib
    _lib._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            _lib.load(missing)
    finally:
        _lib._lib = saved


def test_scan_workspace_checks(lib):
    """The scan needs the workspace it reports; a missing, short, misaligned or
    overlapping one is refused before anything is enqueued."""
    d = dims(batch=2, dim=8, dstate=16, seqlen=64)
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(d), ctypes.byref(need)) == _lib.SSM_OK
    assert need.value >= 256
    ws = P[10]
    assert scan(lib, d) == _lib.SSM_ERR_WORKSPACE                               # none
    assert scan(lib, d, ws=ws, ws_bytes=need.value - 1) == _lib.SSM_ERR_WORKSPACE
    assert scan(lib, d, ws=ws + 16, ws_bytes=need.value) == _lib.SSM_ERR_WORKSPACE
    assert scan(lib, d, ws=P[0], ws_bytes=need.value) == _lib.SSM_ERR_ALIAS     # == u
    assert scan(lib, d, ws=P[8] + 256, ws_bytes=need.value) == _lib.SSM_ERR_ALIAS  # inside y
    # an empty sequence needs none
    d0 = dims(batch=2, dim=8, dstate=16, seqlen=0)
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(d0), ctypes.byref(need)) == _lib.SSM_OK
    assert need.value == 0


@pytest.mark.parametrize("N,ch", [(1, 128), (2, 128), (4, 128), (8, 128), (16, 64)])
def test_scan_workspace_size_formula(lib, N, ch):
    """256-byte header, one flag per channel group, one carried state per group
    (a group is the channels one CTA scans together)."""
    batch, dim = 3, 200
    d = dims(batch=batch, dim=dim, dstate=N, seqlen=10)
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(d), ctypes.byref(need)) == _lib.SSM_OK
    groups = batch * -(-dim // ch)
    r256 = lambda x: -(-x // 256) * 256
    assert need.value == 256 + r256(groups * 4) + r256(groups * ch * N * 4)


def bwd_need(lib, **kw):
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_bwd_workspace_size(ctypes.byref(dims(**kw)), ctypes.byref(need)) == _lib.SSM_OK
    return need.value


@pytest.mark.parametrize("batch,dim,N,L,chunk,nchunks", [
    (4, 5120, 16, 4096, 0, 1),          # Mamba-2.8B layer: a full grid, one chunk
    (8, 1536, 16, 2048, 0, 1),          # Mamba-130M layer: below 8192 tokens
    (1, 1024, 16, 1 << 20, 0, 72),      # DNA-like: 64 CTAs -> 4608 / 64 chunks
    (1, 32, 4, 1 << 18, 0, 128),        # 1 CTA: chunks of the 2048-token minimum
    (2, 40, 16, 4001, 200, 18),         # 200 -> 224 tokens per chunk
    (2, 40, 16, 4001, 4001, 1),         # chunk >= seqlen: one chunk
    (1, 8, 1, 1 << 31, 32, 65473),      # chunks of 32800 tokens: at most 65535 (grid z)
])
def test_bwd_chunk_plan(lib, batch, dim, N, L, chunk, nchunks):
    """The backward's workspace: the checkpoints (batch, dim, ceil(L / 8), N)
    fp32, plus six (nchunks, batch, dim, N) fp32 arrays when the sequence is
    cut into chunks (the states before the chunks, the adjoints into them and
    the chunks' maps), each rounded up to 16 bytes."""
    r16 = lambda x: -(-x // 16) * 16
    ckpt = r16(batch * dim * -(-L // 8) * N * 4)
    arr = r16(nchunks * batch * dim * N * 4) if nchunks > 1 else 0
    assert bwd_need(lib, batch=batch, dim=dim, dstate=N, seqlen=L, chunk=chunk) == ckpt + 6 * arr


def test_bwd_ex_option_checks(lib):
    """ssm_scan_bwd_ex rejects an unknown input term and a gradient type that
    is neither fp32 nor the I/O type, before looking at any pointer."""
    d = dims(io=_lib.SSM_IO_F32)
    def bwd_ex(term, gio, d=d):
        return lib.ssm_scan_bwd_ex(ctypes.byref(d), *P[:8], 1, P[8], None, None, term, gio,
                                   *([None] * 9), None, 0, None)
    assert bwd_ex(2, _lib.SSM_IO_F32) == _lib.SSM_ERR_BAD_OPTION
    assert bwd_ex(_lib.SSM_INPUT_DELTA_B, _lib.SSM_IO_BF16) == _lib.SSM_ERR_BAD_DTYPE
    assert bwd_ex(_lib.SSM_INPUT_DELTA_B, 7, d=dims(io=_lib.SSM_IO_BF16)) == _lib.SSM_ERR_BAD_DTYPE


def test_noalloc_refuses_problems_beyond_its_buffer(lib):
    """The allocation-free scan rejects, on the host, any problem whose scratch
    would not fit its built-in buffer; bad sizes get the usual errors."""
    cap = lib.ssm_scan_fwd_noalloc_max_scratch()
    assert cap == 4 << 20
    big = dims(batch=4, dim=64 * 2000, dstate=16, seqlen=128)   # 8000 groups x 4 KiB of state
    need = ctypes.c_size_t(0)
    assert lib.ssm_scan_fwd_workspace_size(ctypes.byref(big), ctypes.byref(need)) == _lib.SSM_OK
    assert need.value > cap

    def noalloc(d):
        return lib.ssm_scan_fwd_noalloc(ctypes.byref(d) if d is not None else None, P[0], P[1],
                                        P[2], P[3], P[4], P[5], P[6], P[7], 1, P[8], P[9], None)
    assert noalloc(big) == _lib.SSM_ERR_TOO_LARGE
    assert noalloc(None) == _lib.SSM_ERR_NULL_ARG
    assert noalloc(dims(dstate=3)) == _lib.SSM_ERR_UNSUPPORTED_N
    assert noalloc(dims(batch=0)) == _lib.SSM_ERR_BAD_DIMS


def scan_ex(lib, d, opts, **kw):
    a = dict(u=P[0], delta=P[1], A=P[2], B=P[3], C=P[4], D=P[5], z=P[6], bias=P[7], y=P[8],
             last=P[9])
    a.update(kw)
    return lib.ssm_scan_fwd_ex(ctypes.byref(d), None if opts is None else ctypes.byref(opts),
                               a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                               a["bias"], 1, a["y"], a["last"], None, 0, None)


def test_scan_ex_option_checks(lib):
    """ssm_scan_fwd_ex refuses options out of range, a convolution without
    taps, and an initial state or convolution output that overlaps an output,
    before anything is enqueued."""
    d = dims(batch=2, dim=8, dstate=16, seqlen=64)
    O = _lib.ssm_scan_opts
    assert scan_ex(lib, d, O(input_term=2)) == _lib.SSM_ERR_BAD_OPTION
    assert scan_ex(lib, d, O(input_term=-1)) == _lib.SSM_ERR_BAD_OPTION
    assert scan_ex(lib, d, O(conv_width=5)) == _lib.SSM_ERR_BAD_OPTION
    assert scan_ex(lib, d, O(conv_width=-1)) == _lib.SSM_ERR_BAD_OPTION
    assert scan_ex(lib, d, O(conv_width=4)) == _lib.SSM_ERR_NULL_ARG          # no taps
    assert scan_ex(lib, d, O(h0=P[10] + 2)) == _lib.SSM_ERR_MISALIGNED
    assert scan_ex(lib, d, O(h0=P[8])) == _lib.SSM_ERR_ALIAS                  # h0 == y
    assert scan_ex(lib, d, O(h0=P[9] + 64)) == _lib.SSM_ERR_ALIAS             # h0 straddles last_state
    assert scan_ex(lib, d, O(conv_width=4, conv_weight=P[11], u_out=P[8])) == _lib.SSM_ERR_ALIAS
    assert scan_ex(lib, d, O(conv_width=4, conv_weight=P[11], u_out=P[1])) == _lib.SSM_ERR_ALIAS
    assert scan_ex(lib, d, O(conv_width=4, conv_weight=P[11] + 1)) == _lib.SSM_ERR_MISALIGNED
    # the workspace is still checked (these options are all valid)
    ok = O(input_term=_lib.SSM_INPUT_ZOH, conv_width=4, conv_weight=P[11], h0=P[9])
    assert scan_ex(lib, d, ok) == _lib.SSM_ERR_WORKSPACE
