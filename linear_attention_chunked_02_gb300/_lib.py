"""ctypes loader for libkda_solve_tril.so (the C ABI in include/kda_solve_tril.h).

There is no fallback: if the library is missing this raises, so nothing can
silently run anywhere but the CUDA kernels.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkda_solve_tril.so")

# (name, restype, argtypes) for every function the header declares
_c = ctypes
SIGNATURES = [
    ("kda_solve_tril_workspace_size", _c.c_size_t, [_c.c_int64, _c.c_int64, _c.c_int32, _c.c_int32]),
    ("kda_solve_tril_select", _c.c_int, [_c.c_int64, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_size_t]),
    ("kda_solve_tril", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_int64,
                                  _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("kda_solve_tril_ex", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_int64,
                                     _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p, _c.c_size_t, _c.c_void_p,
                                     _c.c_int32, _c.POINTER(_c.c_int32)]),
    ("kda_solve_tril_host", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_int64,
                                       _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                       _c.c_void_p, _c.c_size_t, _c.c_void_p]),
    ("kda_solve_tril_split_static", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64,
                                               _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p]),
    ("kda_solve_tril_prec", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_int64,
                                       _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p]),
    ("kda_solve_tril_bt", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32, _c.c_int64, _c.c_int64,
                                     _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_void_p]),
    ("kda_solve_tril_kgb", _c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_int32,
                                      _c.c_int64, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                      _c.c_void_p]),
    ("kda_selftest_wait", _c.c_int, [_c.c_int32, _c.c_uint32, _c.c_void_p]),
    ("kda_status_string", _c.c_char_p, [_c.c_int32]),
    ("kda_device_error", _c.c_int, [_c.c_int32, _c.POINTER(_c.c_uint32)]),
    ("kda_version", _c.c_int32, []),
]

_LIB = None


def lib() -> ctypes.CDLL:
    """Load the library once; raise if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with linear_attention_chunked_02_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB
