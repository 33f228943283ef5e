"""ctypes binding of libssmscan.so (declarations in include/ssm_scan.h).

Argument marshalling only: every step of the scan runs in the CUDA kernels of
the library.  There is no fallback: if the library cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libssmscan.so")

SSM_F32, SSM_BF16 = 0, 1
SSM_BC_TIME_VARYING, SSM_BC_PER_CHANNEL = 0, 1
STATUS = {
    0: "SSM_OK", -1: "SSM_ERR_NULL", -2: "SSM_ERR_DIMS", -3: "SSM_ERR_ALIGN",
    -4: "SSM_ERR_UNSUPPORTED", -5: "SSM_ERR_CUDA", -6: "SSM_ERR_OVERLAP",
    -7: "SSM_ERR_NOMEM", -8: "SSM_ERR_DEVICE", -9: "SSM_ERR_TIMEOUT",
    -10: "SSM_ERR_SCRATCH",
}
SSM_OK = 0
SSM_ERR_SCRATCH = -10
SSM_NOALLOC_SCRATCH_BYTES = 16 << 20  # include/ssm_scan.h
# names as declared in include/ssm_scan.h
EXPORTS = ("ssm_selective_scan_fwd", "ssm_conv_selective_scan_fwd", "ssm_selective_scan_bwd",
           "ssm_selective_scan_fwd_noalloc",
           "ssm_check_status", "ssm_status_string",
           "ssm_release_workspace", "ssm_workspace_reserved_bytes", "ssm_kernel_launches", "ssm_set_option",
           "ssm_profile_enable", "ssm_profile_read",
           # include/ssm_ssd.h
           "ssm_ssd_fwd")


class SsmDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("dim", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("bc_layout", ctypes.c_int32),
                ("delta_softplus", ctypes.c_int32), ("state_in", ctypes.c_int32),
                ("bbar_mode", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SsdDims(ctypes.Structure):
    """ssm_ssd_dims of include/ssm_ssd.h."""
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64),
                ("nheads", ctypes.c_int64), ("headdim", ctypes.c_int64),
                ("ngroups", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("dt_softplus", ctypes.c_int32),
                ("state_in", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class SSMError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        name = STATUS.get(code, str(code))
        super().__init__(f"{name}: {status_string(code)}" + (f" ({what})" if what else ""))


_lib = None
_lock = threading.Lock()


def lib():
    """Load libssmscan.so (building it first if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                try:
                    from . import build as _build
                    _build.build()
                except Exception as e:  # no silent fallback: the CUDA library is required
                    raise RuntimeError(f"libssmscan.so is missing and could not be built: {e}") from e
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.ssm_selective_scan_fwd.restype = i32
            L.ssm_selective_scan_fwd.argtypes = [vp] * 10 + [ctypes.POINTER(SsmDims), vp]
            L.ssm_conv_selective_scan_fwd.restype = i32
            L.ssm_conv_selective_scan_fwd.argtypes = [vp] * 13 + [ctypes.POINTER(SsmDims), vp]
            L.ssm_selective_scan_bwd.restype = i32
            L.ssm_selective_scan_bwd.argtypes = [vp] * 20 + [ctypes.POINTER(SsmDims), vp]
            L.ssm_selective_scan_fwd_noalloc.restype = i32
            L.ssm_selective_scan_fwd_noalloc.argtypes = [vp] * 10 + [ctypes.POINTER(SsmDims), vp]
            L.ssm_ssd_fwd.restype = i32
            L.ssm_ssd_fwd.argtypes = [vp] * 10 + [ctypes.POINTER(SsdDims), vp]
            L.ssm_check_status.restype = i32
            L.ssm_check_status.argtypes = [vp]
            L.ssm_status_string.restype = ctypes.c_char_p
            L.ssm_status_string.argtypes = [i32]
            L.ssm_release_workspace.restype = i32
            L.ssm_release_workspace.argtypes = []
            L.ssm_workspace_reserved_bytes.restype = i64
            L.ssm_workspace_reserved_bytes.argtypes = []
            L.ssm_kernel_launches.restype = ctypes.c_uint64
            L.ssm_kernel_launches.argtypes = []
            L.ssm_set_option.restype = i32
            L.ssm_set_option.argtypes = [ctypes.c_char_p, i64]
            L.ssm_profile_enable.restype = i32
            L.ssm_profile_enable.argtypes = [i32]
            L.ssm_profile_read.restype = i32
            L.ssm_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p),
                                           ctypes.POINTER(ctypes.c_int64),
                                           ctypes.POINTER(ctypes.c_double), i32]
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().ssm_status_string(int(code)).decode()


def call_fwd(x, delta, A, B, C, D, z, delta_bias, out, final_state, dims: SsmDims,
             stream, noalloc: bool = False) -> int:
    """Raw call: every tensor argument is an integer address (0 = NULL).  With
    ``noalloc`` the call goes to ssm_selective_scan_fwd_noalloc."""
    fn = lib().ssm_selective_scan_fwd_noalloc if noalloc else lib().ssm_selective_scan_fwd
    return fn(x or None, delta or None, A or None, B or None, C or None, D or None,
              z or None, delta_bias or None, out or None, final_state or None,
              ctypes.byref(dims), stream or None)


def call_conv_fwd(x, conv_w, conv_b, conv_state, delta, A, B, C, D, z, delta_bias, out,
                  final_state, dims: SsmDims, stream) -> int:
    """Raw call of ssm_conv_selective_scan_fwd (integer addresses, 0 = NULL)."""
    return lib().ssm_conv_selective_scan_fwd(
        x or None, conv_w or None, conv_b or None, conv_state or None, delta or None, A or None,
        B or None, C or None, D or None, z or None, delta_bias or None, out or None,
        final_state or None, ctypes.byref(dims), stream or None)


def call_bwd(addrs, dims: SsmDims, stream) -> int:
    """Raw call of ssm_selective_scan_bwd: ``addrs`` holds the 20 tensor addresses in
    declaration order (0 = NULL)."""
    assert len(addrs) == 20
    return lib().ssm_selective_scan_bwd(*[a or None for a in addrs], ctypes.byref(dims), stream or None)


def call_ssd(x, dt, A, B, C, D, z, dt_bias, out, final_state, dims: SsdDims, stream) -> int:
    """Raw call of ssm_ssd_fwd (integer addresses, 0 = NULL)."""
    return lib().ssm_ssd_fwd(x or None, dt or None, A or None, B or None, C or None, D or None,
                             z or None, dt_bias or None, out or None, final_state or None,
                             ctypes.byref(dims), stream or None)


def check_status(stream=0) -> int:
    return lib().ssm_check_status(stream or None)


def release_workspace() -> int:
    return lib().ssm_release_workspace()


def workspace_reserved_bytes() -> int:
    n = int(lib().ssm_workspace_reserved_bytes())
    if n < 0:
        raise SSMError(n, "ssm_workspace_reserved_bytes")
    return n


def kernel_launches() -> int:
    return int(lib().ssm_kernel_launches())


def set_option(name: str, value: int) -> None:
    rc = lib().ssm_set_option(name.encode(), int(value))
    if rc != SSM_OK:
        raise SSMError(rc, f"option {name}={value}")


def profile_enable(on: bool) -> None:
    lib().ssm_profile_enable(1 if on else 0)


def profile_read(max_rows: int = 8) -> dict:
    names = (ctypes.c_char_p * max_rows)()
    launches = (ctypes.c_int64 * max_rows)()
    ms = (ctypes.c_double * max_rows)()
    n = lib().ssm_profile_read(names, launches, ms, max_rows)
    if n < 0:
        raise SSMError(n, "ssm_profile_read")
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(min(n, max_rows))}
