"""ctypes view of libssm_scan.so (declared in include/ssm_scan.h).

Loading fails loudly when the library has not been built; there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# The library built in-tree.  SSM_SCAN_LIBRARY may name another build of the
# same sources, e.g. the -DSSM_DEBUG build (build.build(debug=True)).
LIBRARY = os.environ.get("SSM_SCAN_LIBRARY") or os.path.join(HERE, "libssm_scan.so")

# ssm_status codes (include/ssm_scan.h)
SSM_OK = 0
SSM_ERR_NULL_ARG = -1
SSM_ERR_BAD_DIMS = -2
SSM_ERR_UNSUPPORTED_N = -3
SSM_ERR_BAD_DTYPE = -4
SSM_ERR_MISALIGNED = -5
SSM_ERR_CUDA = -6
SSM_ERR_WORKSPACE = -7
SSM_ERR_ALIAS = -8
SSM_ERR_TIMEOUT = -9
SSM_ERR_TOO_LARGE = -10
SSM_ERR_BAD_OPTION = -11
SSM_ERR_DEVICE = -12

SSM_INPUT_DELTA_B = 0
SSM_INPUT_ZOH = 1

SSM_IO_F32 = 0
SSM_IO_BF16 = 1

# every symbol include/ssm_scan.h declares
EXPORTS = ("ssm_build_id", "ssm_probe_ex2", "ssm_scan_bwd", "ssm_scan_bwd_ex",
           "ssm_scan_bwd_workspace_size", "ssm_scan_fwd",
           "ssm_scan_fwd_ex", "ssm_scan_fwd_host", "ssm_scan_fwd_noalloc",
           "ssm_scan_fwd_noalloc_max_scratch", "ssm_scan_fwd_noalloc_status",
           "ssm_scan_fwd_status", "ssm_scan_fwd_workspace_size", "ssm_state_step",
           "ssm_status_string", "ssm_version")


class ssm_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("io", ctypes.c_int32), ("chunk", ctypes.c_int32)]


class ssm_scan_opts(ctypes.Structure):
    _fields_ = [("input_term", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("h0", ctypes.c_void_p), ("conv_weight", ctypes.c_void_p),
                ("conv_bias", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("u_out", ctypes.c_void_p), ("wait_limit", ctypes.c_int32),
                ("test_skip_handoff", ctypes.c_int32)]


class SSMError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load(path: str = LIBRARY) -> ctypes.CDLL:
    """Load the library once.  Raises if it is missing: build it first."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing; build it with "
            "`python -m selective_state_space_116_b300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    dims_p = ctypes.POINTER(ssm_dims)
    lib.ssm_scan_fwd.restype = i32
    lib.ssm_scan_fwd.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    lib.ssm_scan_fwd_ex.restype = i32
    lib.ssm_scan_fwd_ex.argtypes = [dims_p, ctypes.POINTER(ssm_scan_opts), vp, vp, vp, vp, vp, vp,
                                    vp, vp, i32, vp, vp, vp, sz, vp]
    lib.ssm_scan_fwd_status.restype = i32
    lib.ssm_scan_fwd_status.argtypes = [vp, sz, vp]
    lib.ssm_scan_fwd_noalloc_status.restype = i32
    lib.ssm_scan_fwd_noalloc_status.argtypes = [vp]
    lib.ssm_scan_bwd.restype = i32
    lib.ssm_scan_bwd.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp,
                                 vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssm_scan_bwd_ex.restype = i32
    lib.ssm_scan_bwd_ex.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, i32, i32,
                                    vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.ssm_scan_bwd_workspace_size.restype = i32
    lib.ssm_scan_bwd_workspace_size.argtypes = [dims_p, ctypes.POINTER(sz)]
    lib.ssm_scan_fwd_host.restype = i32
    lib.ssm_scan_fwd_host.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    lib.ssm_scan_fwd_noalloc.restype = i32
    lib.ssm_scan_fwd_noalloc.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp]
    lib.ssm_scan_fwd_noalloc_max_scratch.restype = sz
    lib.ssm_scan_fwd_noalloc_max_scratch.argtypes = []
    lib.ssm_scan_fwd_workspace_size.restype = i32
    lib.ssm_scan_fwd_workspace_size.argtypes = [dims_p, ctypes.POINTER(sz)]
    lib.ssm_state_step.restype = i32
    lib.ssm_state_step.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp]
    lib.ssm_probe_ex2.restype = i32
    lib.ssm_probe_ex2.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp]
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_status_string.argtypes = [i32]
    lib.ssm_version.restype = i32
    lib.ssm_version.argtypes = []
    lib.ssm_build_id.restype = ctypes.c_char_p
    lib.ssm_build_id.argtypes = []
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().ssm_status_string(int(status)).decode()
