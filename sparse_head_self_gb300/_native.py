"""ctypes loader for libfibatt.so (argument types only; no computation here).

The library must have been built (``__graft_entry__.build()`` or
``python sparse_head_self_gb300/build.py``); loading fails loudly otherwise.
There is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from .build import LIB, LIB_CHECKS, ROOT

HEADER = os.path.join(ROOT, "include", "fibatt.h")

OK = 0
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "CUDA", 4: "OOM"}
F32, BF16 = 0, 1

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_ip = ctypes.POINTER(ctypes.c_int)

_SIGS = {
    "fibatt_wythoff_row": (ctypes.c_int, [ctypes.c_int64, _i64p, _i64p]),
    "fibatt_wythoff_row_modified": (ctypes.c_int, [ctypes.c_int64, _i64p, _i64p]),
    "fibatt_window_schedule": (ctypes.c_int, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, _i64p]),
    "fibatt_support_build": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _i64p, _i64p, _i64p,
                                            ctypes.c_int, ctypes.POINTER(_vp)]),
    "fibatt_support_build_distances": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _i32p, _i32p,
                                                      ctypes.c_int, ctypes.POINTER(_vp)]),
    "fibatt_support_set_global_token": (ctypes.c_int, [_vp, ctypes.c_int]),
    "fibatt_support_info": (ctypes.c_int, [_vp, _ip, _ip, _ip]),
    "fibatt_support_get": (ctypes.c_int, [_vp, _i32p, _i32p, _i64p]),
    "fibatt_support_destroy": (None, [_vp]),
    "fibatt_fwd": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                  ctypes.c_float, _vp, _vp, _vp]),
    "fibatt_bwd_workspace_bytes": (ctypes.c_size_t, [_vp, ctypes.c_int]),
    "fibatt_bwd": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                  _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, ctypes.c_size_t,
                                  _vp]),
    "fibatt_bwd_noalloc": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp, _vp,
                                          _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]),
    "fibatt_last_error": (ctypes.c_char_p, []),
    "fibatt_version": (ctypes.c_char_p, []),
    "fibatt_launch_count": (ctypes.c_uint64, []),
    "fibatt_device_error": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_uint)]),
}


class FibattError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libfibatt {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


def header_functions() -> list[str]:
    """Names of every function include/fibatt.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fibatt_\w+)\s*\(", text)))


def lib():
    """The loaded libfibatt (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libfibatt is not built ({path} missing); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def check(status: int) -> None:
    if status != OK:
        raise FibattError(status, lib().fibatt_last_error().decode())


def lib_path() -> str:
    """The library this process loads: the checks build (bounds-checked
    kernels) when FIBATT_CHECKS=1 is set, else the regular one."""
    return LIB_CHECKS if os.environ.get("FIBATT_CHECKS") == "1" else LIB
