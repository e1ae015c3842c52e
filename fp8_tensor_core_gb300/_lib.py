"""ctypes loader for the in-tree CUDA library ``_build/libfp8g.so``.

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfp8g.so")

# Symbols declared in include/fp8g.h, with their ctypes signatures.
_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64


class Scales(ctypes.Structure):
    """fp8g_scales: output scales and block scales (NULL pointers: absent)."""
    _fields_ = [("out_a", ctypes.c_void_p), ("out_a_len", ctypes.c_int64),
                ("out_b", ctypes.c_void_p), ("out_b_len", ctypes.c_int64),
                ("block_a", ctypes.c_void_p), ("block_a_ld", ctypes.c_int64),
                ("block_b", ctypes.c_void_p), ("block_b_ld", ctypes.c_int64),
                ("block_k", ctypes.c_int32)]


class Epilogue(ctypes.Structure):
    """fp8g_epilogue: D = round(act(alpha * value + beta * C + bias))."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("c", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("activation", ctypes.c_int32), ("round_mode", ctypes.c_int32)]


class Plan(ctypes.Structure):
    """fp8g_plan: the launch the library would make for a problem."""
    _fields_ = [(name, ctypes.c_int32) for name in ("kernel", "tile_n", "stages", "stream_k", "mma_issuers",
                                                     "shared_sm", "token_box", "grid", "k_split")]


_scales_p = ctypes.POINTER(Scales)
_epi_p = ctypes.POINTER(Epilogue)
SIGNATURES = {
    "fp8_gemm_nt": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_grouped_masked": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                               _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_nt_scaled": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                          ctypes.c_int, ctypes.c_int, _c_void_p, _i64, _c_void_p,
                                          _i64, ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_grouped_masked_scaled": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                                      _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                                      ctypes.c_int, _c_void_p, _i64, _c_void_p, _i64,
                                                      ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_nt_blockscaled": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                               ctypes.c_int, ctypes.c_int, _c_void_p, _i64, _c_void_p,
                                               _i64, ctypes.c_int, ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_grouped_masked_blockscaled": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                                           _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
                                                           ctypes.c_int, _c_void_p, _i64, _c_void_p,
                                                           _i64, ctypes.c_int, ctypes.c_uint32,
                                                           _c_void_p]),
    "fp8_gemm_nt_ex": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64, ctypes.c_int,
                                      ctypes.c_int, _scales_p, _epi_p, ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_grouped_masked_ex": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                                  _i64, _i64, ctypes.c_int, ctypes.c_int, _scales_p, _epi_p,
                                                  ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_grouped_contiguous": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                                   _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_uint32,
                                                   _c_void_p]),
    "fp8_gemm_grouped_contiguous_ex": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                                      _i64, _i64, ctypes.c_int, ctypes.c_int, _scales_p, _epi_p,
                                                      ctypes.c_uint32, _c_void_p]),
    "fp8_gemm_nt_noalloc": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                           ctypes.c_int, ctypes.c_int, _c_void_p]),
    "fp8g_get_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _c_void_p]),
    "fp8g_init": (ctypes.c_int, [_i64, _c_void_p]),
    "fp8g_release_stream": (ctypes.c_int, [_c_void_p]),
    "fp8g_describe_plan": (ctypes.c_int, [ctypes.c_int, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_uint32,
                                          ctypes.c_int, ctypes.c_int, ctypes.POINTER(Plan)]),
    "fp8g_shutdown": (ctypes.c_int, []),
    "fp8g_set_wait_timeout_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "fp8g_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fp8g_version": (ctypes.c_int, []),
}

_lock = threading.Lock()
_lib = None


class LibraryNotBuilt(RuntimeError):
    pass


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise LibraryNotBuilt(
                "fp8g CUDA library not built (%s missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib
