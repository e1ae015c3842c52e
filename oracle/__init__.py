"""CPU oracle for the FP8 GEMM path -- TEST INFRASTRUCTURE, not the product.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It shares no code with the CUDA library
and never calls it.  The arithmetic lives in ``fp8_oracle.c`` (plain C,
fp64); this module compiles it with gcc on first use and wraps it for numpy.

What it computes, with its sources:

* ``decode_fp8`` / ``decode_table`` -- FP8 code to exact double.  E4M3 is
  4 exponent + 3 mantissa bits and E5M2 is 5 + 2 ("DeepGEMM：基于 Hopper
  Tensor Core 的 FP8 矩阵乘法内核优化实践", §3.1); the biases, NaN and
  infinity codes are the OCP FP8 reading (the page gives only the bit split).
* ``gemm_nt`` -- D = A·Bᵀ with FP8 inputs, exact products, double
  accumulation in ascending k, one BF16 round-to-nearest-even (same page,
  §1.3: FP8 inputs, FP32 accumulation; BF16 output is the plainest reading of
  its BF16 back-end remark).
* ``gemm_grouped_masked`` -- the masked grouped variant: only rows
  m < masked_m[g] of each group are computed or written ("一次“转置”，半张
  算力：DeepSeek SwapAB 漂流史", §3.1 and §3.3, valid_m).
* ``gemm_grouped_contiguous`` -- groups' token rows concatenated along M,
  group g owning rows offsets[g]..offsets[g+1]-1 and multiplying B[g].
* ``epilogue`` -- round_mode(act(alpha*S + beta*C + bias)) of exact sums S,
  BF16 rounding to nearest even / toward zero / toward +inf / toward -inf
  (DeepGEMM page §3.3: fused alpha, beta, bias, ReLU and rounding mode).
* ``gemm_blockscaled`` -- every product scaled by the UE8M0 factors of its
  K group (32 or 128 elements) for its A row and B row, then summed and
  rounded once (DeepGEMM page §5.2 per-128-element groups; SwapAB page §5,
  UE8M0 scales on SM100, and §3.4, scale factors in the Blackwell MMA).
* ``gemm_nt_scaled`` / ``gemm_grouped_masked_scaled`` -- the same products
  multiplied back by per-tensor or per-channel FP32 scales before the one
  rounding (DeepGEMM page §3.1 and §5.2).
* ``check_bf16`` -- the acceptance rule for a GPU result:
  |gpu - oracle| <= ulp_bf16(oracle) + 1e-6 * sum_k |a_k b_k| per element.

Pins (tests marked "not gpu") tie every function to something other than
itself: torch's float8/bfloat16 conversions, exact rational brute force,
closed forms for structured matrices, and printed fixtures.
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
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile ``fp8_oracle.c`` into ``_build/liboracle.so`` (plain -O2, no
    fast-math, no contraction of separately rounded operations)."""
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
        lib.oracle_decode_fp8.restype = ctypes.c_double
        lib.oracle_decode_fp8.argtypes = [ctypes.c_uint8, ctypes.c_int]
        lib.oracle_decode_table.restype = None
        lib.oracle_decode_table.argtypes = [ctypes.c_int, _f64p]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_default_threads.restype = ctypes.c_int
        lib.oracle_default_threads.argtypes = []
        lib.oracle_gemm_nt.restype = None
        lib.oracle_gemm_nt.argtypes = [_u8p, _u8p, _i64, _i64, _i64,
                                       ctypes.c_int, ctypes.c_int, _u16p,
                                       _f64p, _f64p, ctypes.c_int]
        lib.oracle_gemm_nt_entries.restype = None
        lib.oracle_gemm_nt_entries.argtypes = [_u8p, _u8p, _i64, ctypes.c_int,
                                               ctypes.c_int, _i64p, _i64p,
                                               _i64, _u16p, _f64p, _f64p]
        lib.oracle_gemm_grouped_masked.restype = None
        lib.oracle_gemm_grouped_masked.argtypes = [
            _u8p, _u8p, _i32p, _i64, _i64, _i64, _i64, ctypes.c_int,
            ctypes.c_int, _u16p, _f64p, ctypes.c_int]
        _f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_gemm_nt_scaled.restype = None
        lib.oracle_gemm_nt_scaled.argtypes = [_u8p, _u8p, _i64, _i64, _i64, ctypes.c_int,
                                              ctypes.c_int, _f32p, _i64, _f32p, _i64, _u16p,
                                              _f64p, ctypes.c_int]
        lib.oracle_gemm_grouped_masked_scaled.restype = None
        lib.oracle_gemm_grouped_masked_scaled.argtypes = [
            _u8p, _u8p, _i32p, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _f32p, _i64,
            _f32p, _i64, _u16p, _f64p, ctypes.c_int]
        lib.oracle_gemm_blockscaled.restype = None
        lib.oracle_gemm_blockscaled.argtypes = [
            _u8p, _u8p, _i32p, _i64, _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _u8p, _i64,
            _u8p, _i64, _i64, _u16p, _f64p, _f64p, _f64p, ctypes.c_int]
        lib.oracle_gemm_grouped_contiguous.restype = None
        lib.oracle_gemm_grouped_contiguous.argtypes = [_u8p, _u8p, _i32p, _i64, _i64, _i64, _i64, ctypes.c_int,
                                                       ctypes.c_int, _u16p, _f64p, _f64p, ctypes.c_int]
        lib.oracle_round_bf16_mode.restype = ctypes.c_uint16
        lib.oracle_round_bf16_mode.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.oracle_epilogue.restype = None
        lib.oracle_epilogue.argtypes = [_f64p, _f64p, _i64, _i64, _i64, _i32p, ctypes.c_double,
                                        ctypes.c_double, _u16p, _f32p, ctypes.c_int, ctypes.c_int,
                                        _u16p, _f64p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray, t):
    if a is None:
        return ctypes.cast(None, t)
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


def default_threads() -> int:
    """Cores the oracle's thread pool uses when ``nthreads <= 0``."""
    return int(_load().oracle_default_threads())


def decode_fp8(code: int, fmt: int) -> float:
    return float(_load().oracle_decode_fp8(code & 0xFF, fmt))


def decode_table(fmt: int) -> np.ndarray:
    out = np.empty(256, np.float64)
    _load().oracle_decode_table(fmt, _ptr(out, _f64p))
    return out


def round_bf16(x: float) -> int:
    return int(_load().oracle_round_bf16(float(x)))


def round_bf16_array(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(x, np.float64).ravel()
    return np.array([lib.oracle_round_bf16(float(v)) for v in flat],
                    np.uint16).reshape(np.shape(x))


def bf16_to_double(h: int) -> float:
    return float(_load().oracle_bf16_to_double(h & 0xFFFF))


def bf16_bits_to_f64(h: np.ndarray) -> np.ndarray:
    """Vectorised exact BF16 -> double (a BF16 code is the top half of the
    binary32 with the same value)."""
    h = np.asarray(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_nt(A: np.ndarray, B: np.ndarray, fa: int = E4M3, fb: int = E4M3,
            want_exact: bool = False, nthreads: int = 0):
    """Dense oracle. A: uint8 [M,K], B: uint8 [N,K] (K contiguous).
    Returns (D_bf16 uint16 [M,N], absdot float64 [M,N][, exact float64])."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    D = np.empty((M, N), np.uint16)
    absdot = np.empty((M, N), np.float64)
    exact = np.empty((M, N), np.float64) if want_exact else None
    _load().oracle_gemm_nt(_ptr(A, _u8p), _ptr(B, _u8p), M, N, K, fa, fb,
                           _ptr(D, _u16p), _ptr(exact, _f64p),
                           _ptr(absdot, _f64p), int(nthreads))
    if want_exact:
        return D, absdot, exact
    return D, absdot


def gemm_nt_entries(A: np.ndarray, B: np.ndarray, ms, ns, fa: int = E4M3,
                    fb: int = E4M3):
    """Selected dense outputs D[ms[i], ns[i]] (for sampled checks of
    full-size problems).  Returns (bf16 codes, absdot, exact)."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    K = A.shape[1]
    assert B.shape[1] == K
    ms = np.ascontiguousarray(ms, np.int64)
    ns = np.ascontiguousarray(ns, np.int64)
    assert ms.shape == ns.shape
    assert ms.size == 0 or (ms.min() >= 0 and ms.max() < A.shape[0])
    assert ns.size == 0 or (ns.min() >= 0 and ns.max() < B.shape[0])
    cnt = ms.size
    D = np.empty(cnt, np.uint16)
    absdot = np.empty(cnt, np.float64)
    exact = np.empty(cnt, np.float64)
    _load().oracle_gemm_nt_entries(_ptr(A, _u8p), _ptr(B, _u8p), K, fa, fb,
                                   _ptr(ms, _i64p), _ptr(ns, _i64p), cnt,
                                   _ptr(D, _u16p), _ptr(exact, _f64p),
                                   _ptr(absdot, _f64p))
    return D, absdot, exact


def gemm_grouped_masked(A: np.ndarray, B: np.ndarray, masked_m: np.ndarray,
                        D_init: np.ndarray, fa: int = E4M3, fb: int = E4M3,
                        nthreads: int = 0):
    """Masked grouped oracle.  A: uint8 [G,M_max,K], B: uint8 [G,N,K],
    masked_m: int32 [G] in [0, M_max], D_init: uint16 [G,M_max,N] (copied;
    rows m >= masked_m[g] keep these bits).  Returns (D, absdot) where
    absdot is 0 on rows that are not computed."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    assert G == G2 and K == K2
    mm = np.ascontiguousarray(masked_m, np.int32)
    assert mm.shape == (G,) and (mm.size == 0 or (mm.min() >= 0 and mm.max() <= M_max))
    D = np.array(D_init, np.uint16, copy=True, order="C")
    assert D.shape == (G, M_max, N)
    absdot = np.zeros((G, M_max, N), np.float64)
    _load().oracle_gemm_grouped_masked(_ptr(A, _u8p), _ptr(B, _u8p),
                                       _ptr(mm, _i32p), G, M_max, N, K, fa, fb,
                                       _ptr(D, _u16p), _ptr(absdot, _f64p),
                                       int(nthreads))
    return D, absdot


def gemm_nt_scaled(A: np.ndarray, B: np.ndarray, scale_a: np.ndarray, scale_b: np.ndarray,
                   fa: int = E4M3, fb: int = E4M3, nthreads: int = 0):
    """Scaled dense oracle: D[m,n] = bf16(sa(m) sb(n) sum_k a b) with FP32
    scales of length 1 (per tensor) or M / N (per row / per column).
    Returns (D_bf16, absdot_scaled)."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    sa = np.ascontiguousarray(scale_a, np.float32).ravel()
    sb = np.ascontiguousarray(scale_b, np.float32).ravel()
    assert sa.size in (1, M) and sb.size in (1, N)
    D = np.empty((M, N), np.uint16)
    absdot = np.empty((M, N), np.float64)
    f32p = ctypes.POINTER(ctypes.c_float)
    _load().oracle_gemm_nt_scaled(_ptr(A, _u8p), _ptr(B, _u8p), M, N, K, fa, fb,
                                  _ptr(sa, f32p), sa.size, _ptr(sb, f32p), sb.size,
                                  _ptr(D, _u16p), _ptr(absdot, _f64p), int(nthreads))
    return D, absdot


def gemm_grouped_masked_scaled(A: np.ndarray, B: np.ndarray, masked_m: np.ndarray,
                               scale_a: np.ndarray, scale_b: np.ndarray, D_init: np.ndarray,
                               fa: int = E4M3, fb: int = E4M3, nthreads: int = 0):
    """Scaled masked grouped oracle; scale_a has G or G*M_max entries,
    scale_b G or G*N.  Rows m >= masked_m[g] keep D_init's bits."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    assert G == G2 and K == K2
    mm = np.ascontiguousarray(masked_m, np.int32)
    sa = np.ascontiguousarray(scale_a, np.float32).ravel()
    sb = np.ascontiguousarray(scale_b, np.float32).ravel()
    assert sa.size in (G, G * M_max) and sb.size in (G, G * N)
    D = np.array(D_init, np.uint16, copy=True, order="C")
    absdot = np.zeros((G, M_max, N), np.float64)
    f32p = ctypes.POINTER(ctypes.c_float)
    _load().oracle_gemm_grouped_masked_scaled(_ptr(A, _u8p), _ptr(B, _u8p), _ptr(mm, _i32p), G,
                                              M_max, N, K, fa, fb, _ptr(sa, f32p), sa.size,
                                              _ptr(sb, f32p), sb.size, _ptr(D, _u16p),
                                              _ptr(absdot, _f64p), int(nthreads))
    return D, absdot


def gemm_blockscaled(A: np.ndarray, B: np.ndarray, sfa: np.ndarray, sfb: np.ndarray,
                     gran: int = 128, masked_m=None, D_init=None, fa: int = E4M3, fb: int = E4M3,
                     nthreads: int = 0, want_exact: bool = False, want_accbound: bool = False):
    """Block-scaled oracle.  Dense: A [M,K], B [N,K], sfa [KS,lda], sfb
    [KS,ldb] uint8 UE8M0 codes (KS = ceil(K/gran), row m of A scaled by
    sfa[k // gran, m]).  Grouped: A [G,M_max,K], B [G,N,K], sfa [G,KS,lda],
    sfb [G,KS,ldb], masked_m [G] (rows m >= masked_m[g] keep D_init's bits).
    Returns (D_bf16, absdot[, exact sums][, accbound]): accbound = 2^-23 *
    sum |S_i| over the running sums S_i at the ends of the 32-element K
    slices, the bound on the error of an FP32 accumulator that adds each
    tensor-core instruction's result with at most one FP32 ulp of error
    (the acc_bound term of check_bf16)."""
    dense = np.ndim(A) == 2
    A3 = np.ascontiguousarray(A, np.uint8).reshape((1,) + np.shape(A) if dense else np.shape(A))
    B3 = np.ascontiguousarray(B, np.uint8).reshape((1,) + np.shape(B) if dense else np.shape(B))
    G, M_max, K = A3.shape
    G2, N, K2 = B3.shape
    assert G == G2 and K == K2 and gran in (32, 128)
    KS = -(-K // gran)
    SA = np.ascontiguousarray(sfa, np.uint8).reshape(G, KS, -1)
    SB = np.ascontiguousarray(sfb, np.uint8).reshape(G, KS, -1)
    lda, ldb = SA.shape[2], SB.shape[2]
    assert lda >= M_max and ldb >= N
    if masked_m is not None:
        mm = np.ascontiguousarray(masked_m, np.int32)
        assert mm.shape == (G,) and (mm.size == 0 or (mm.min() >= 0 and mm.max() <= M_max))
        mm_p = _ptr(mm, _i32p)
    else:
        mm_p = None
    if D_init is None:
        D = np.zeros((G, M_max, N), np.uint16)
    else:
        D = np.array(D_init, np.uint16, copy=True, order="C").reshape(G, M_max, N)
    absdot = np.zeros((G, M_max, N), np.float64)
    exact = np.zeros((G, M_max, N), np.float64)
    accb = np.zeros((G, M_max, N), np.float64)
    _load().oracle_gemm_blockscaled(_ptr(A3, _u8p), _ptr(B3, _u8p), mm_p, G, M_max, N, K, fa, fb,
                                    _ptr(SA, _u8p), lda, _ptr(SB, _u8p), ldb, gran, _ptr(D, _u16p),
                                    _ptr(exact, _f64p), _ptr(absdot, _f64p), _ptr(accb, _f64p), int(nthreads))
    out = (D, absdot) + ((exact,) if want_exact else ()) + ((accb,) if want_accbound else ())
    if dense:
        out = tuple(x[0] for x in out)
    return out


def gemm_grouped_contiguous(A: np.ndarray, B: np.ndarray, offsets: np.ndarray, D_init=None, fa: int = E4M3,
                            fb: int = E4M3, nthreads: int = 0, want_exact: bool = False):
    """Contiguous grouped oracle: A uint8 [M_total, K] (groups' token rows
    concatenated), B uint8 [G, N, K], offsets int32 [G+1] (group g owns rows
    offsets[g] .. offsets[g+1]-1).  Rows outside every group keep D_init's
    bits.  Returns (D, absdot[, exact])."""
    A = np.ascontiguousarray(A, np.uint8)
    B = np.ascontiguousarray(B, np.uint8)
    M_total, K = A.shape
    G, N, K2 = B.shape
    assert K == K2
    off = np.ascontiguousarray(offsets, np.int32)
    assert off.shape == (G + 1,) and np.all(np.diff(off) >= 0) and off[0] >= 0 and off[-1] <= M_total
    D = np.zeros((M_total, N), np.uint16) if D_init is None else np.array(D_init, np.uint16, copy=True, order="C")
    exact = np.zeros((M_total, N), np.float64)
    absdot = np.zeros((M_total, N), np.float64)
    _load().oracle_gemm_grouped_contiguous(_ptr(A, _u8p), _ptr(B, _u8p), _ptr(off, _i32p), G, M_total, N, K, fa,
                                           fb, _ptr(D, _u16p), _ptr(exact, _f64p), _ptr(absdot, _f64p),
                                           int(nthreads))
    return (D, absdot, exact) if want_exact else (D, absdot)


ROUND_RN, ROUND_RZ, ROUND_RU, ROUND_RD = 0, 1, 2, 3


def round_bf16_mode(x: float, mode: int) -> int:
    """BF16 code of x rounded in direction `mode` (0 nearest-even, 1 toward
    zero, 2 toward +inf, 3 toward -inf)."""
    return int(_load().oracle_round_bf16_mode(float(x), int(mode)))


def epilogue(S: np.ndarray, absS: np.ndarray, alpha: float = 1.0, beta: float = 0.0, C=None, bias=None,
             relu: bool = False, mode: int = ROUND_RN, masked_m=None, D_init=None):
    """Fused-epilogue oracle: round_mode(act(alpha*S + beta*C + bias[g, n]))
    per element.  S, absS: exact sums and sum|terms| shaped [M,N] or
    [G,M_max,N]; C: BF16 codes shaped like S (or None); bias: float32 [N] or
    [G,N] (or None); masked rows keep D_init's bits.  Returns (D, absdot)."""
    S = np.ascontiguousarray(S, np.float64)
    absS = np.ascontiguousarray(absS, np.float64)
    shape = S.shape
    S3 = S.reshape((1,) + shape if S.ndim == 2 else shape)
    G, M_max, N = S3.shape
    Cc = None if C is None else np.ascontiguousarray(C, np.uint16).reshape(S3.shape)
    bb = None if bias is None else np.ascontiguousarray(bias, np.float32).reshape(G, N)
    mm = None if masked_m is None else np.ascontiguousarray(masked_m, np.int32)
    D = (np.zeros(S3.shape, np.uint16) if D_init is None
         else np.array(D_init, np.uint16, copy=True, order="C").reshape(S3.shape))
    absdot = np.zeros(S3.shape, np.float64)
    _load().oracle_epilogue(_ptr(S3, _f64p), _ptr(absS.reshape(S3.shape), _f64p), G * M_max, M_max, N,
                            _ptr(mm, _i32p), float(alpha), float(beta), _ptr(Cc, _u16p),
                            _ptr(bb, ctypes.POINTER(ctypes.c_float)), 1 if relu else 0, int(mode),
                            _ptr(D, _u16p), _ptr(absdot, _f64p))
    return D.reshape(shape), absdot.reshape(shape)


# ---- acceptance rule -------------------------------------------------------

REL_TOL = 1e-6   # coefficient of sum_k |a_k b_k| in the per-element bound


def ulp_bf16(ref_bits: np.ndarray) -> np.ndarray:
    """Spacing of the binade of each BF16 value: 2^(floor(log2|x|) - 7) for
    normal x, 2^-133 for subnormal x, 0 for x == 0."""
    h = np.asarray(ref_bits, np.uint16).astype(np.int64)
    e = (h >> 7) & 0xFF
    m = h & 0x7F
    out = np.where(e > 0, np.ldexp(1.0, (e - 134).astype(np.int32)), 0.0)
    out = np.where((e == 0) & (m != 0), np.ldexp(1.0, -133), out)
    return out


def check_bf16(gpu_bits: np.ndarray, ref_bits: np.ndarray,
               absdot: np.ndarray, rel: float = REL_TOL, acc_bound=None):
    """Per-element acceptance: |gpu - ref| <= ulp_bf16(ref) + rel*absdot
    (+ acc_bound, the accumulation-order bound gemm_blockscaled returns for
    block-scaled products).  NaN or infinity on either side fails.  Returns
    (ok, report dict)."""
    g = bf16_bits_to_f64(gpu_bits)
    r = bf16_bits_to_f64(ref_bits)
    tol = ulp_bf16(ref_bits) + rel * np.asarray(absdot, np.float64)
    if acc_bound is not None:
        tol = tol + np.asarray(acc_bound, np.float64)
    diff = np.abs(g - r)
    finite = np.isfinite(g) & np.isfinite(r)
    bad = (~finite) | (diff > tol)
    nbad = int(np.count_nonzero(bad))
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio = np.where(tol > 0, diff / tol, np.where(diff > 0, np.inf, 0.0))
    ratio = np.where(finite, ratio, np.inf)
    worst = float(ratio.max()) if ratio.size else 0.0
    exact = int(np.count_nonzero(np.asarray(gpu_bits) == np.asarray(ref_bits)))
    rep = {"n": int(np.size(g)), "bad": nbad, "worst_ratio": worst,
           "bit_exact": exact}
    if nbad:
        idx = np.flatnonzero(bad.ravel())[:8]
        rep["first_bad"] = [(int(i), float(g.ravel()[i]), float(r.ravel()[i]),
                             float(tol.ravel()[i])) for i in idx]
    return nbad == 0, rep
