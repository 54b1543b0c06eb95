"""ctypes view of the C ABI in include/msda.h (libmsda.so, built in-tree).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
# MSDA_LIBRARY points the binding at another build of the same library
LIB_PATH = os.environ.get("MSDA_LIBRARY") or os.path.join(PKG, "libmsda.so")

MSDA_OK = 0
STATUS_NAMES = {0: "MSDA_OK", 1: "MSDA_ERR_INVALID_ARG", 2: "MSDA_ERR_UNSUPPORTED", 3: "MSDA_ERR_MISALIGNED",
                4: "MSDA_ERR_WORKSPACE", 5: "MSDA_ERR_CUDA"}
ACCUM = {"auto": 0, "native": 1, "fp32": 2, "deterministic": 3}
ACCUM_NAMES = {v: k for k, v in ACCUM.items()}
BWD_ACCUMULATE = 1
BWD_WORKSPACE_ZEROED = 2
KERNEL_NAMES = {0: "forward", 1: "backward", 2: "zero", 3: "convert", 4: "tile_count", 5: "tile_scan",
                6: "tile_place", 7: "tile_accum", 8: "touch_count"}


class MsdaError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


class TraceRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int), ("ms", ctypes.c_float), ("work", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def _declare(lib):
    i64, vp, c_int, c_uint, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    dims = [i64] * 7
    lib.msda_forward.argtypes = [c_int] + dims + [vp] * 6 + [vp]
    lib.msda_forward.restype = c_int
    lib.msda_backward.argtypes = [c_int, c_int, c_uint] + dims + [vp] * 9 + [vp, sz, vp]
    lib.msda_backward.restype = c_int
    lib.msda_forward_fused.argtypes = [c_int] + dims + [vp] * 7 + [vp]
    lib.msda_forward_fused.restype = c_int
    lib.msda_backward_fused.argtypes = [c_int, c_int, c_uint] + dims + [vp] * 11 + [vp, sz, vp]
    lib.msda_backward_fused.restype = c_int
    lib.msda_reduction_ceiling.argtypes = [c_int, c_int, c_int, c_int, vp, sz, ctypes.POINTER(ctypes.c_double), vp]
    lib.msda_reduction_ceiling.restype = c_int
    lib.msda_backward_workspace_size.argtypes = [c_int, c_int] + dims
    lib.msda_backward_workspace_size.restype = sz
    lib.msda_resolve_accum.argtypes = [c_int, c_int] + dims
    lib.msda_resolve_accum.restype = c_int
    lib.msda_last_error.restype = ctypes.c_char_p
    lib.msda_status_string.argtypes = [c_int]
    lib.msda_status_string.restype = ctypes.c_char_p
    lib.msda_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), c_int]
    lib.msda_device_errors.restype = c_int
    lib.msda_version.restype = c_int
    lib.msda_trace_enable.argtypes = [c_int]
    lib.msda_trace_enable.restype = c_int
    lib.msda_trace_pause.argtypes = [c_int]
    lib.msda_trace_pause.restype = None
    lib.msda_trace_read.argtypes = [ctypes.POINTER(TraceRecord), c_int, ctypes.POINTER(c_int)]
    lib.msda_trace_read.restype = c_int
    lib.msda_kernel_name.argtypes = [c_int]
    lib.msda_kernel_name.restype = ctypes.c_char_p
    return lib


def lib():
    """The loaded library (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; build it with `python -m scale_deformable_attention_gb300.build` "
                    "(needs nvcc for sm_103a). There is no CPU fallback.")
            # load torch first so the library binds to the CUDA runtime torch already loaded
            import torch  # noqa: F401
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def check(status: int):
    if status != MSDA_OK:
        msg = lib().msda_last_error().decode(errors="replace")
        raise MsdaError(status, msg)
