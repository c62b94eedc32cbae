"""ctypes declarations of the C ABI in include/fp4mx.h.

The library is loaded from ``lib/libfp4mx.so`` inside this package (built by
``_build.build()``). A missing or unloadable library raises -- there is no
fallback implementation of any step.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

from . import _build

_lock = threading.Lock()
_lib = None


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL_PTR = 1
    ERR_SHAPE = 2
    ERR_GROUP = 3
    ERR_UNSUPPORTED = 4
    ERR_INDEX = 5
    ERR_CUDA = 6
    ERR_POINTER = 7
    ERR_ALIAS = 8
    ERR_ALIGN = 9
    ERR_TIMEOUT = 10


# Every function the header declares, with its ctypes signature.
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
SIGNATURES = {
    "fp4_mx_unpack": ([_vp, _vp, _vp, _i64, _i64, _vp], ctypes.c_int),
    "fp4_nv_embedding_gather": ([_vp, _i64, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp],
                                ctypes.c_int),
    "fp4_nv_dequant": ([_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp], ctypes.c_int),
    "fp4_mx_quantize": ([_vp, _vp, _vp, _i64, _i64, _vp], ctypes.c_int),
    "fp4_mx_unpack_pages": ([_vp, _i64, _vp, _vp, _i64, _i64, _vp, _vp, _vp], ctypes.c_int),
    "fp4_mx_moe_gemm": ([_vp, _vp, _i64, _i64, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp],
                        ctypes.c_int),
    "fp4_mx_moe_forward": ([_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _i64, _i64,
                            _vp, _i64, _vp, _vp, _vp], ctypes.c_int),
    "fp4_mx_moe_workspace_bytes": ([_i64, _i64, _i64, _i64, _i64], ctypes.c_int64),
    "fp4_mx_moe_forward_noalloc": ([_vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                    _i64, _i64, _vp, _vp, _vp], ctypes.c_int),
    "fp4_mx_moe_static_scratch_bytes": ([], ctypes.c_int64),
    "fp4_wait_selftest": ([ctypes.c_int32, _vp, _vp], ctypes.c_int),
    "fp4_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "fp4_last_error": ([], ctypes.c_char_p),
    "fp4_abi_version": ([], ctypes.c_int),
}


def library_path() -> str:
    return _build.LIBRARY


def load(build_if_missing: bool = True):
    """Load (building first if needed and allowed) the CUDA library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIBRARY
        if build_if_missing and _build.is_stale():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; run __graft_entry__.build() "
                "(nvcc for sm_103a). There is no CPU fallback.")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().fp4_status_string(int(code)).decode()


def last_error() -> str:
    return load().fp4_last_error().decode()
