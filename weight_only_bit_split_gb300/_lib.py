"""ctypes loader for libwobs.so (the C ABI in include/wobs.h).

The library is built in-tree (``python -m weight_only_bit_split_gb300.build``
or ``__graft_entry__.build()``).  There is no fallback: if it is missing or
fails to load, every entry point raises.
"""
import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwobs.so")

_lock = threading.Lock()
_lib = None

c_int, c_int64, c_size_t, c_void_p = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
c_float_p = ctypes.POINTER(ctypes.c_float)

# name -> (restype, argtypes); must match include/wobs.h
SIGNATURES = {
    "wobs_last_error": (ctypes.c_char_p, []),
    "wobs_version": (c_int, []),
    "wobs_bw_probe": (c_int, [c_void_p, c_size_t, c_int, c_int, c_void_p, c_void_p]),
    "wobs_gemv_f16": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int, c_void_p, c_int, c_int,
                              c_void_p, c_size_t, c_void_p]),
    "wobs_gemv_bf16": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int, c_void_p, c_void_p,
                               c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_gemv_bf16_noalloc": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int, c_void_p,
                                       c_void_p, c_int, c_int, c_void_p]),
    "wobs_quantize_q8_1": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_void_p]),
    "wobs_quantize_q4_0": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "wobs_quantize_nf4": (c_int, [c_void_p, c_int64, c_int, c_int, c_float_p, c_void_p, c_void_p,
                                  c_void_p]),
    "wobs_gemv_q4_0_q8_1": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                    c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_gemv_q4_0_f32": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_gemv_q8_0_f32": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_quantize_q8_0": (c_int, [c_void_p, c_int64, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "wobs_gemv_q8_0_q8_1": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                    c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_gemv_nf4": (c_int, [c_void_p, c_void_p, c_float_p, c_void_p, c_int64, c_int, c_void_p,
                              c_void_p, c_int, c_int, c_void_p, c_size_t, c_void_p]),
    "wobs_dequantize_nf4": (c_int, [c_void_p, c_void_p, c_float_p, c_int, c_int, c_void_p, c_int64,
                                    c_void_p]),
    "wobs_argmax": (c_int, [c_int, c_void_p, c_int64, c_int, c_int, c_void_p, c_void_p, c_size_t,
                            c_void_p]),
    "wobs_argmin": (c_int, [c_int, c_void_p, c_int64, c_int, c_int, c_void_p, c_void_p, c_size_t,
                            c_void_p]),
    "wobs_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int]),
    "wobs_q4_0_q8_1_blockdots": (c_int, [c_void_p, c_void_p, c_int, c_int, c_int, c_void_p,
                                         c_void_p]),
    "wobs_error_word": (c_int, [c_void_p, ctypes.POINTER(c_int)]),
    "wobs_selftest_wait_timeout": (c_int, [ctypes.c_longlong, c_void_p]),
}


class LibraryMissing(RuntimeError):
    pass


def get():
    """The loaded library (loads it on first use; raises if unavailable)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise LibraryMissing(
                    f"{LIB_PATH} not found: build it with "
                    "`python -m weight_only_bit_split_gb300.build` (no CPU fallback exists)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
