"""Seeded synthetic inputs shared by the oracle's tests and the GPU path's
tests and bench.  It holds none of the GEMM arithmetic: it maps
(seed, element index) to an FP8 byte through SplitMix64, an optional
Box-Muller normal, and a round-to-nearest-even, saturating FP8 encoder.
The C source is ``synth.c``; this module compiles it with gcc on first use.

Workload recipes (one function per input of each workload) live at the
bottom; every seed is ``0x0F8C0DE + 1000*workload + run`` plus a small tensor
index, so the same workload always gets the same bytes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
        "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
        "-o", tmp, _SRC, "-lm", "-lpthread"])
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.synth_splitmix64_at.restype = ctypes.c_uint64
        lib.synth_splitmix64_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_uniform_at.restype = ctypes.c_double
        lib.synth_uniform_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_normal_at.restype = ctypes.c_double
        lib.synth_normal_at.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_encode_fp8.restype = ctypes.c_uint8
        lib.synth_encode_fp8.argtypes = [ctypes.c_double, ctypes.c_int]
        for name in ("synth_fill_uniform_fp8", "synth_fill_normal_fp8"):
            f = getattr(lib, name)
            f.restype = None
            f.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, ctypes.c_uint64,
                          ctypes.c_double, ctypes.c_double, ctypes.c_int,
                          ctypes.c_int]
        lib.synth_fill_uniform_int.restype = None
        lib.synth_fill_uniform_int.argtypes = [_i32p, ctypes.c_int64,
                                               ctypes.c_uint64, ctypes.c_int32,
                                               ctypes.c_int32]
        lib.synth_fill_u16.restype = None
        lib.synth_fill_u16.argtypes = [_u16p, ctypes.c_int64, ctypes.c_uint64]
        _lib = lib
        return lib


def splitmix64_at(seed: int, i: int) -> int:
    return int(_load().synth_splitmix64_at(seed & (2**64 - 1), i))


def uniform_at(seed: int, i: int) -> float:
    return float(_load().synth_uniform_at(seed & (2**64 - 1), i))


def normal_at(seed: int, i: int) -> float:
    return float(_load().synth_normal_at(seed & (2**64 - 1), i))


def encode_fp8(x: float, fmt: int) -> int:
    return int(_load().synth_encode_fp8(float(x), fmt))


def encode_fp8_array(x, fmt: int) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, np.float64).ravel()
    return np.array([lib.synth_encode_fp8(float(v), fmt) for v in flat],
                    np.uint8).reshape(np.shape(x))


def uniform_fp8(shape, seed: int, lo: float, hi: float, fmt: int = E4M3,
                first: int = 0, nthreads: int = 0) -> np.ndarray:
    """FP8 codes of U[lo,hi) samples for elements [first, first+prod(shape))
    of the stream `seed`."""
    out = np.empty(shape, np.uint8)
    _load().synth_fill_uniform_fp8(out.ctypes.data_as(_u8p), int(first),
                                   int(out.size), seed & (2**64 - 1),
                                   float(lo), float(hi), fmt, int(nthreads))
    return out


def normal_fp8(shape, seed: int, mean: float, std: float, fmt: int = E4M3,
               first: int = 0, nthreads: int = 0) -> np.ndarray:
    """FP8 codes of N(mean, std^2) samples for elements [first, first+n)."""
    out = np.empty(shape, np.uint8)
    _load().synth_fill_normal_fp8(out.ctypes.data_as(_u8p), int(first),
                                  int(out.size), seed & (2**64 - 1),
                                  float(mean), float(std), fmt, int(nthreads))
    return out


def uniform_int(n: int, seed: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    _load().synth_fill_uniform_int(out.ctypes.data_as(_i32p), int(n),
                                   seed & (2**64 - 1), int(lo), int(hi))
    return out


def u16_pattern(shape, seed: int) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    _load().synth_fill_u16(out.ctypes.data_as(_u16p), int(out.size),
                           seed & (2**64 - 1))
    return out


# ---- workload recipes -----------------------------------------------------

SEED_BASE = 0x0F8C0DE


def seed_for(workload: int, run: int = 0, tensor: int = 0) -> int:
    return SEED_BASE + 1000 * workload + run + 100 * tensor


def rows_fp8(kind: str, shape, seed: int, fmt: int, row_first: int = 0,
             nthreads: int = 0, **kw) -> np.ndarray:
    """Rows [row_first, row_first+shape[0]) of a 2-D tensor whose full width
    is shape[-1] (rows are contiguous in the element counter)."""
    first = row_first * int(np.prod(shape[1:]))
    if kind == "uniform":
        return uniform_fp8(shape, seed, kw["lo"], kw["hi"], fmt, first, nthreads)
    if kind == "normal":
        return normal_fp8(shape, seed, kw.get("mean", 0.0), kw["std"], fmt,
                          first, nthreads)
    raise ValueError(kind)
