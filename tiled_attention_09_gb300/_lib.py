"""ctypes loader for libfa.so: argument and return types of every C entry point.

Marshalling only. Loading fails loudly (RuntimeError) when the library has not
been built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

c_int, c_float, c_size_t, c_void_p, c_uint = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_uint
c_longlong = ctypes.c_longlong

STATUS_NAMES = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_ALIGNMENT",
    4: "FA_ERR_WORKSPACE",
    5: "FA_ERR_CUDA",
    6: "FA_ERR_TIMEOUT",
    7: "FA_ERR_DEVICE_FAULT",
}
FA_F16, FA_BF16 = 0, 1


class FAOptions(ctypes.Structure):
    """struct fa_options of include/fa.h."""
    _fields_ = [("n_kv_heads", c_int), ("kv_len", c_void_p), ("o_fp32", c_int), ("dq_mode", c_int)]


# (name, restype, argtypes) for every symbol declared in include/fa.h and include/fa_selftest.h
SIGNATURES = [
    ("fa_fwd", c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_float, c_int,
                       c_int, c_void_p]),
    ("fa_fwd_ex", c_int, [c_void_p] * 6 + [c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_void_p]),
    ("fa_fwd_opt", c_int, [c_void_p] * 6 + [c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                            ctypes.POINTER(FAOptions), c_void_p]),
    ("fa_bwd_workspace_size", c_size_t, [c_int, c_int, c_int, c_int]),
    ("fa_fwd_split", c_int, [c_void_p] * 6 + [c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                              ctypes.POINTER(FAOptions), c_int, c_void_p, c_size_t, c_void_p]),
    ("fa_fwd_kv_splits", c_int, [c_int] * 5),
    ("fa_fwd_tiles_per_item", c_int, [c_int] * 5),
    ("fa_fwd_workspace_size", c_size_t, [c_int] * 5),
    ("fa_bwd", c_int, [c_void_p] * 10 + [c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                         c_void_p]),
    ("fa_bwd_opt", c_int, [c_void_p] * 10 + [c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                             ctypes.POINTER(FAOptions), c_void_p]),
    ("fa_bwd_noalloc", c_int, [c_void_p] * 10 + [c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_void_p]),
    ("fa_bwd_preprocess", c_int, [c_void_p] * 5 + [c_size_t, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    ("fa_bwd_main", c_int, [c_void_p] * 7 + [c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                             c_void_p]),
    ("fa_bwd_dq_convert", c_int, [c_void_p, c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_float, c_int,
                                  c_void_p]),
    ("fa_bwd_preprocess_opt", c_int, [c_void_p] * 5 + [c_size_t] + [c_int] * 6 + [ctypes.POINTER(FAOptions),
                                                                                 c_void_p]),
    ("fa_bwd_main_opt", c_int, [c_void_p] * 7 + [c_void_p, c_size_t, c_int, c_int, c_int, c_int, c_float, c_int,
                                                 c_int, ctypes.POINTER(FAOptions), c_void_p]),
    ("fa_bwd_uses_dq_pass", c_int, [c_int, c_int, ctypes.POINTER(FAOptions)]),
    ("fa_bwd_dq_pass", c_int, [c_void_p] * 6 + [c_size_t, c_int, c_int, c_int, c_int, c_float, c_int, c_int,
                                                ctypes.POINTER(FAOptions), c_void_p]),
    ("fa_decode_splits", c_int, [c_int] * 5),
    ("fa_decode_workspace_size", c_size_t, [c_int] * 8),
    ("fa_decode", c_int, [c_void_p] * 7 + [c_void_p, c_size_t] + [c_int] * 9 + [c_float, c_int, c_int, c_void_p]),
    ("fa_device_status", c_int, [c_void_p, ctypes.POINTER(c_uint)]),
    ("fa_status_string", ctypes.c_char_p, [c_int]),
    ("fa_set_wait_timeout_ns", None, [ctypes.c_ulonglong]),
    ("fa_version", c_int, []),
    ("fa_selftest_mma_rate", c_int, [c_int, c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    ("fa_selftest_mma_pattern", c_int, [c_int] * 8 + [c_void_p, c_void_p]),
    ("fa_selftest_gemm", c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_void_p]),
    ("fa_selftest_wait_timeout", c_int, [ctypes.c_ulonglong, c_void_p]),
    ("fa_selftest_ex2_rate", c_int, [c_int, c_int, c_void_p, c_void_p]),
    ("fa_selftest_block_order", c_int, [c_int, c_int, c_longlong, c_void_p, c_void_p]),
    ("fa_selftest_copy", c_int, [c_void_p, c_void_p, c_size_t, c_int, c_void_p]),
]

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")


def lib_path() -> str:
    return LIB_PATH


def load():
    """Return the loaded library, raising RuntimeError if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libfa.so is not built ({LIB_PATH} missing); run `python -m tiled_attention_09_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def check(fn: str, code: int):
    if code != 0:
        raise FAError(fn, code)
