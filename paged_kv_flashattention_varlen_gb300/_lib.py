"""ctypes view of libpattn.so (the C ABI declared in include/pattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of the library. Loading fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpattn.so")

# Exported functions and their (restype, argtypes).
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)
SIGNATURES = {
    "pattn_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "pattn_forward_append": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                  _f, _i, _vp]),
    "pattn_forward_fp8qk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "pattn_quantize_qk": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                               _i, _vp]),
    "pattn_workspace_size_fp8qk": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "pattn_forward_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "pattn_quantize_v": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "pattn_workspace_size_fp8": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "pattn_forward_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i,
                                   _vp]),
    "pattn_forward_host": (_i, [_vp, _vp, _vp, _sz, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                _f, _i, _vp]),
    "pattn_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "pattn_set_workspace": (_i, [_vp, _sz]),
    "pattn_get_device_status": (_i, [_vp]),
    "pattn_selftest_wait_timeout": (_i, [_vp]),
    "pattn_selftest_attention_timeout": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                              _f, _i, _vp]),
    "pattn_plan_items": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _i, _vp, _vp]),
    "pattn_status_string": (ctypes.c_char_p, [_i]),
    "pattn_profile_enable": (_i, [_i]),
    "pattn_profile_read": (_i, [_dp, _dp, _dp, _ip]),
    "pattn_profile_read_kernels": (_i, [_dp, _ip]),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load libpattn.so (built by ``paged_kv_flashattention_varlen_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"libpattn.so not found at {LIB_PATH}: build it first "
                    "(python -m paged_kv_flashattention_varlen_gb300.build); there is no fallback")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
