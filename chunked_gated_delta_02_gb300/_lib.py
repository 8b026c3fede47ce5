"""ctypes loader of libkda.so and the argument types of its C ABI (include/kda.h).

There is no fallback: if the shared library is missing or fails to load, every
call raises. Build it with ``python -c "import __graft_entry__ as g; g.build()"``
or ``python -m chunked_gated_delta_02_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkda.so")
_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float

STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_WORKSPACE",
          4: "KDA_ERR_CUDA", 5: "KDA_ERR_DEVICE_STATUS"}

# name -> (restype, argtypes)
SIGNATURES = {
    "kda_fwd_workspace_size": (ctypes.c_size_t, [I, I, I, I, I, I]),
    "kda_fwd_workspace_size_ex": (ctypes.c_size_t, [I, I, I, I, I, I, I, ctypes.c_uint32]),
    "kda_fwd": (I, [P, P, P, P, P, P, P, F, F, P, P, P, I, I, I, I, I, I, P, P, ctypes.c_size_t, P]),
    "kda_fwd_with_events": (I, [P, P, P, P, P, P, P, F, F, P, P, P, I, I, I, I, I, I, P, P, ctypes.c_size_t, P,
                                 P]),
    "kda_fwd_ex": (I, [P, P, P, P, P, P, P, F, F, P, P, P, I, I, I, I, I, I, ctypes.c_uint32, P, P, ctypes.c_size_t,
                        P, P]),
    "kda_fwd_noalloc": (I, [P, P, P, P, P, P, P, F, F, P, P, P, I, I, I, I, I, I, P, P]),
    "kda_debug_chunk_matrices": (I, [P, P, P, P, P, P, F, P, I, I, I, I, I, P, P, ctypes.c_size_t, P]),
    "kda_max_chunks": (ctypes.c_int64, [I, I, I]),
    "kda_fwd_plan": (I, [I, I, I, I, I, I, I, ctypes.c_uint32, ctypes.POINTER(I), ctypes.POINTER(I)]),
    "kda_status_string": (ctypes.c_char_p, [I]),
    "kda_get_device_status": (I, [P, ctypes.POINTER(ctypes.c_int)]),
    "kda_debug_wait_timeout": (I, [ctypes.c_longlong, P]),
    "kda_version": (I, []),
}


class KDAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = lib().kda_status_string(code).decode() if code in STATUS else "unknown"
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({msg})")


def lib():
    """The loaded libkda.so (raises OSError if it is not built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise OSError(f"libkda.so not found at {LIB_PATH}; build it first "
                                  "(python -m chunked_gated_delta_02_gb300.build)")
                h = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(h, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = h
    return _lib


def check(fn: str, code: int):
    if code != 0:
        raise KDAError(fn, code)
