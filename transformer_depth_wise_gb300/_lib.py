"""ctypes binding of libattnres.so (argument marshalling only).

The names and argument orders mirror include/attnres.h one for one.  The
library is loaded from this package directory; if it is missing, every call
raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattnres.so")

ATTNRES_F32 = 0
ATTNRES_BF16 = 1
ATTNRES_MAX_SOURCES = 256
ATTNRES_MAX_QUERIES = 64

STATUS = {
    0: "ATTNRES_OK",
    -1: "ATTNRES_ERR_NULL",
    -2: "ATTNRES_ERR_SHAPE",
    -3: "ATTNRES_ERR_DTYPE",
    -4: "ATTNRES_ERR_ALIGNMENT",
    -5: "ATTNRES_ERR_TOO_MANY_SOURCES",
    -6: "ATTNRES_ERR_CUDA",
    -7: "ATTNRES_ERR_CAPACITY",
    -8: "ATTNRES_ERR_VALUE",
    -9: "ATTNRES_ERR_TIMEOUT",
    -10: "ATTNRES_ERR_SCRATCH",
}

# Every symbol include/attnres.h declares, with its ctypes signature.
_vp, _i64, _int, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_pp = ctypes.POINTER(ctypes.c_void_p)
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "attnres_depth_aggregate": (_int, [_pp, _int, _i64, _i64, _i64, _int, _vp, _vp, _f, _vp, _vp, _vp,
                                       _vp]),
    "attnres_block_phase1": (_int, [_pp, _int, _i64, _i64, _i64, _int, _vp, _vp, _int, _f, _vp, _vp,
                                    _vp, _vp]),
    "attnres_block_phase2_merge": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _vp, _f, _vp,
                                          _vp, _vp]),
    "attnres_partial_update": (_int, [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _vp]),
    "attnres_block_merge_update": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _vp, _f,
                                          _vp, _vp, _vp, _vp, _f, _vp, _vp]),
    "attnres_rms_norm": (_int, [_vp, _i64, _i64, _i64, _int, _vp, _f, _vp, _vp]),
    "attnres_depth_aggregate_backward": (_int, [_vp, _int, _i64, _i64, _i64, _int, _vp, _vp, _f, _vp, _vp,
                                                _int, _vp, _vp, _vp, _i64, _vp]),
    "attnres_depth_aggregate_backward_workspace_rows": (_i64, [_i64, _int]),
    "attnres_full_stack_two_phase": (_int, [_vp, _int, _int, _i64, _i64, _i64, _int, _vp, _vp, _vp, _f, _vp,
                                            _vp, _i64, _vp]),
    "attnres_full_stack_two_phase_workspace_bytes": (_i64, [_int, _int, _i64, _i64, _i64, _int]),
    "attnres_depth_aggregate_backward_noalloc": (_int, [_vp, _int, _i64, _i64, _i64, _int, _vp, _vp, _f, _vp,
                                                        _vp, _int, _vp, _vp, _vp]),
    "attnres_full_stack_forward": (_int, [_pp, _int, _i64, _i64, _i64, _int, _vp, _vp, _vp, _f, _vp,
                                          _vp]),
    "attnres_block_schedule": (_int, [_int, _int, _ip, _ip, _int]),
    "attnres_atomic_block_size": (_int, [_int, _int]),
    "attnres_take_device_error": (_int, []),
    "attnres_set_wait_limit": (_int, [_i64]),
    "attnres_status_string": (ctypes.c_char_p, [_int]),
}

_lib = None


class AttnResError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().attnres_status_string(status).decode() if _lib is not None else ""
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({msg})")


def lib() -> ctypes.CDLL:
    """Load libattnres.so (built by transformer_depth_wise_gb300.build); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m transformer_depth_wise_gb300.build` "
                "(the CUDA path has no fallback)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(fn: str, status: int) -> int:
    if status < 0:
        raise AttnResError(fn, status)
    return status


def ptr_array(ptrs) -> ctypes.Array:
    arr = (ctypes.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = p
    return arr
