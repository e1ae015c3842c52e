"""fp8_tensor_core_gb300 -- FP8 GEMM for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/fp8g.h``: it checks dtypes,
shapes, contiguity and devices, then passes raw pointers and the current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or library fallback.

    fp8_gemm_nt(A, B)                        D[M,N] = A[M,K] . B[N,K]^T (BF16)
    fp8_gemm_grouped_masked(A, B, masked_m)  D[g,m,:] for m < masked_m[g]
"""
from __future__ import annotations

import ctypes

from . import _lib

E4M3 = 0
E5M2 = 1
SWAP_AUTO = 0
SWAP_ON = 1
SWAP_OFF = 2
DEBUG_ONE_STAGE = 0x10


WHOLE_TILES = 0x100   # SwapAB kernel: whole tiles per CTA instead of stream-K ranges
STREAM_K = 0x800      # SM-pair dense kernel: stream-K split of the last partial wave
SPLIT_TAIL = 0x80     # SM-pair dense kernel: split the last wave's tiles along K whenever possible
SINGLE_SM_TILES = 0x200   # dense non-swapped: one SM per 128-row tile instead of SM pairs
NO_PDL = 0x400            # launch without programmatic dependent launch
PAIR_TILES = 0x4000       # dense: always SM-pair tiles when M > 128
ONE_MMA_ISSUER = 0x8000   # block-scaled kernels: one MMA-issuing thread
TWO_MMA_ISSUERS = 0x2000  # block-scaled tile kernels: two issuers even with one buffer each
SHARE_SM = 0x1000         # SwapAB kernel: half an SM per CTA (next launch overlaps the drain)
NO_SHARE_SM = 0x40        # SwapAB kernel: never share an SM (default shares it for <= 16 tokens)


def TOKEN_BOX(n: int) -> int:
    """Flag bits: SwapAB token rows per TMA copy (multiple of 16 dividing the chunk)."""
    return ((int(n) // 16) & 15) << 24


def STAGES(n: int) -> int:
    """Flag bits capping the shared-memory pipeline at n stages (1..15)."""
    return (int(n) & 15) << 20


def TILE_N(n: int) -> int:
    """Flag bits forcing an N tile of n (multiple of 32, <= 256) in the
    non-swapped kernel."""
    return ((int(n) // 32) & 15) << 16


DEBUG_DROP_FIRST_LOAD = 0x20

OK = 0
ERR_INVALID_ARG = 1
ERR_MISALIGNED = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_NO_DEVICE = 6
ERR_MASKED_M_RANGE = 7


class Fp8gError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s" % (where, fp8g_status_string(code)))


def fp8g_status_string(code: int) -> str:
    return _lib.load().fp8g_status_string(int(code)).decode()


def fp8g_version() -> int:
    return int(_lib.load().fp8g_version())


def fp8g_init(max_tiles: int = 0, stream=None) -> None:
    """Allocate the stream-K workspace of `stream` (default: the current
    torch stream) on the current device at its largest size (counters for
    max_tiles output tiles, 0 = the library default), so that later calls
    on that stream allocate nothing -- e.g. before capturing a CUDA graph
    from it."""
    rc = _lib.load().fp8g_init(int(max_tiles), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8g_init")


def fp8g_release_stream(stream=None) -> None:
    """Synchronise `stream` (default: the current torch stream) and free its
    stream-K workspace on the current device."""
    rc = _lib.load().fp8g_release_stream(_stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8g_release_stream")


KERNEL_TOKEN_TILES, KERNEL_SM_PAIRS, KERNEL_SWAP_AB = 0, 1, 2
LAYOUT_DENSE, LAYOUT_MASKED, LAYOUT_CONTIGUOUS = 0, 1, 2


def fp8g_describe_plan(layout: int, G: int, rows: int, N: int, K: int, token_hint: int = 0,
                       sf_group_k: int = 0, flags: int = 0, sms: int = 0, smem_optin: int = 0) -> dict:
    """The launch the library would make for a problem (kernel, tile,
    stages, split, issuers, SM sharing, token rows per copy, grid), without
    touching memory; sms / smem_optin 0 plan for the current device."""
    out = _lib.Plan()
    rc = _lib.load().fp8g_describe_plan(int(layout), int(G), int(rows), int(N), int(K), int(token_hint),
                                        int(sf_group_k), int(flags), int(sms), int(smem_optin), ctypes.byref(out))
    if rc != OK:
        raise Fp8gError(rc, "fp8g_describe_plan")
    return {name: int(getattr(out, name)) for name, _ in _lib.Plan._fields_}


def fp8g_shutdown() -> None:
    """Free the library's stream-K workspaces (every stream, every device)."""
    rc = _lib.load().fp8g_shutdown()
    if rc != OK:
        raise Fp8gError(rc, "fp8g_shutdown")


def fp8g_set_wait_timeout_ns(ns: int) -> int:
    return int(_lib.load().fp8g_set_wait_timeout_ns(int(ns)))


def fp8g_get_device_status(stream=None):
    """Synchronise `stream` (default: current), read and clear the device
    status word.  Returns (code, block, role, detail)."""
    import torch
    info = (ctypes.c_int32 * 4)()
    s = _stream_handle(stream)
    rc = _lib.load().fp8g_get_device_status(info, s)
    if rc != OK:
        raise Fp8gError(rc, "fp8g_get_device_status")
    return tuple(int(v) for v in info)


class _NoSwitch:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


_NO_SWITCH = _NoSwitch()


def _on_device(device):
    """Make `device` current for the call (a no-op when it already is)."""
    import torch
    if device.index is None or device.index == torch.cuda.current_device():
        return _NO_SWITCH
    return torch.cuda.device(device)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _fp8_code(t, explicit):
    import torch
    if t.dtype == torch.float8_e4m3fn:
        return E4M3 if explicit is None else explicit
    if t.dtype == torch.float8_e5m2:
        return E5M2 if explicit is None else explicit
    if t.dtype == torch.uint8:
        if explicit is None:
            raise TypeError("uint8 operand needs an explicit FP8 format (E4M3 or E5M2)")
        return explicit
    raise TypeError("operand dtype %s is not an FP8 code type" % t.dtype)


def _check_operand(t, name, ndim):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dim() != ndim:
        raise ValueError("%s must have %d dimensions, got %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous (row-major, K innermost)" % name)


def fp8_gemm_nt(A, B, D=None, a_dtype=None, b_dtype=None, flags: int = 0, stream=None):
    """D[M,N] (bf16) = A[M,K] . B[N,K]^T with FP8 A and B (float8 dtypes, or
    uint8 codes with an explicit format).  Returns D."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 2)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch: A has %d, B has %d" % (K, K2))
    if A.device != B.device:
        raise ValueError("A and B on different devices")
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 2)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N) or D.device != A.device:
            raise ValueError("D must be a contiguous bf16 [M, N] tensor on A's device")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_nt(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                     fa, fb, int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_nt")
    return D


def fp8_gemm_grouped_masked(A, B, masked_m, D=None, max_m_hint: int = 0, a_dtype=None,
                            b_dtype=None, flags: int = 0, stream=None):
    """Masked grouped GEMM: A[G,M_max,K], B[G,N,K], masked_m int32[G] on the
    device.  Rows m < masked_m[g] of D[g] are written; the others are left
    untouched.  Returns D (allocated uninitialised if not given)."""
    import torch
    _check_operand(A, "A", 3)
    _check_operand(B, "B", 3)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    if G != G2 or K != K2:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    if not masked_m.is_cuda or masked_m.dtype != torch.int32 or tuple(masked_m.shape) != (G,) \
            or not masked_m.is_contiguous():
        raise ValueError("masked_m must be a contiguous int32 CUDA tensor of shape [G]")
    if D is None:
        D = torch.empty((G, M_max, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 3)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (G, M_max, N):
            raise ValueError("D must be a contiguous bf16 [G, M_max, N] tensor")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_grouped_masked(
            A.data_ptr(), B.data_ptr(), D.data_ptr(), masked_m.data_ptr(), G, M_max, N, K,
            int(max_m_hint), fa, fb, int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_grouped_masked")
    return D


def fp8_gemm_nt_noalloc(A, B, D, a_dtype=None, b_dtype=None, stream=None):
    """D[M,N] = A[M,K] . B[N,K]^T for M <= 256 tokens without any device
    allocation by the library: stream-K scratch lives in a fixed 32 MiB device
    array inside the library (for callers whose allocator must own all
    device memory, or that cannot take cudaMalloc's synchronisation).  D
    must be given.  Calls on unordered streams race on the shared scratch."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 2)
    _check_operand(D, "D", 2)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2 or D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N):
        raise ValueError("shapes: A [M,K], B [N,K], D bf16 [M,N]")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                             fa, fb, _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_nt_noalloc")
    return D


def _check_scale(t, name, lengths):
    import torch
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.numel() not in lengths:
        raise ValueError("%s must be a contiguous float32 CUDA tensor with %s entries"
                         % (name, " or ".join(str(v) for v in sorted(set(lengths)))))


def fp8_gemm_nt_scaled(A, B, scale_a, scale_b, D=None, a_dtype=None, b_dtype=None, flags: int = 0,
                       stream=None):
    """D[m,n] = bf16(sa(m) * sb(n) * sum_k A[m,k] B[n,k]) with float32 CUDA
    scales: scale_a of 1 (per tensor) or M (per row) entries, scale_b of 1
    or N (per output channel)."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 2)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch: A has %d, B has %d" % (K, K2))
    _check_scale(scale_a, "scale_a", (1, M))
    _check_scale(scale_b, "scale_b", (1, N))
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 2)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N):
            raise ValueError("D must be a contiguous bf16 [M, N] tensor")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_nt_scaled(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, fa, fb,
                                            scale_a.data_ptr(), scale_a.numel(), scale_b.data_ptr(),
                                            scale_b.numel(), int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_nt_scaled")
    return D


def fp8_gemm_grouped_masked_scaled(A, B, masked_m, scale_a, scale_b, D=None, max_m_hint: int = 0,
                                   a_dtype=None, b_dtype=None, flags: int = 0, stream=None):
    """Masked grouped GEMM times scales: scale_a of G (per group) or G*M_max
    (per token row) entries, scale_b of G or G*N (per output channel)."""
    import torch
    _check_operand(A, "A", 3)
    _check_operand(B, "B", 3)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    if G != G2 or K != K2:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    if not masked_m.is_cuda or masked_m.dtype != torch.int32 or tuple(masked_m.shape) != (G,):
        raise ValueError("masked_m must be a contiguous int32 CUDA tensor of shape [G]")
    _check_scale(scale_a, "scale_a", (G, G * M_max))
    _check_scale(scale_b, "scale_b", (G, G * N))
    if D is None:
        D = torch.empty((G, M_max, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 3)
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_grouped_masked_scaled(
            A.data_ptr(), B.data_ptr(), D.data_ptr(), masked_m.data_ptr(), G, M_max, N, K,
            int(max_m_hint), fa, fb, scale_a.data_ptr(), scale_a.numel(), scale_b.data_ptr(),
            scale_b.numel(), int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_grouped_masked_scaled")
    return D


def _check_sf(t, name, groups, ks, rows):
    import torch
    if (not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous() or t.dim() != 3
            or t.shape[0] != groups or t.shape[1] != ks or t.shape[2] < rows or t.shape[2] % 16 != 0):
        raise ValueError("%s must be a contiguous uint8 CUDA tensor [%d, %d, ld] with ld >= %d, ld %% 16 == 0"
                         % (name, groups, ks, rows))


def fp8_gemm_nt_blockscaled(A, B, sf_a, sf_b, D=None, sf_group_k: int = 128, a_dtype=None, b_dtype=None,
                            flags: int = 0, stream=None):
    """Block-scaled D[m,n] = bf16(sum_k A[m,k] B[n,k] 2^(sf_a[k/gs, m]-127)
    2^(sf_b[k/gs, n]-127)).  sf_a: uint8 [ks, lda] (or [1, ks, lda]), sf_b:
    uint8 [ks, ldb]; ks = ceil(K / sf_group_k), lda >= M and ldb >= N
    multiples of 16."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 2)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch: A has %d, B has %d" % (K, K2))
    if sf_group_k not in (32, 128):
        raise ValueError("sf_group_k must be 32 or 128")
    ks = -(-K // sf_group_k)
    sa = sf_a if sf_a.dim() == 3 else sf_a.unsqueeze(0)
    sb = sf_b if sf_b.dim() == 3 else sf_b.unsqueeze(0)
    _check_sf(sa, "sf_a", 1, ks, M)
    _check_sf(sb, "sf_b", 1, ks, N)
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 2)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N):
            raise ValueError("D must be a contiguous bf16 [M, N] tensor")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_nt_blockscaled(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, fa, fb,
                                                 sa.data_ptr(), sa.shape[2], sb.data_ptr(), sb.shape[2],
                                                 int(sf_group_k), int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_nt_blockscaled")
    return D


def fp8_gemm_grouped_masked_blockscaled(A, B, masked_m, sf_a, sf_b, D=None, max_m_hint: int = 0,
                                        sf_group_k: int = 128, a_dtype=None, b_dtype=None, flags: int = 0,
                                        stream=None):
    """Masked grouped GEMM with block scales: sf_a uint8 [G, ks, lda]
    (lda >= M_max), sf_b uint8 [G, ks, ldb] (ldb >= N)."""
    import torch
    _check_operand(A, "A", 3)
    _check_operand(B, "B", 3)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    if G != G2 or K != K2:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    if not masked_m.is_cuda or masked_m.dtype != torch.int32 or tuple(masked_m.shape) != (G,):
        raise ValueError("masked_m must be a contiguous int32 CUDA tensor of shape [G]")
    if sf_group_k not in (32, 128):
        raise ValueError("sf_group_k must be 32 or 128")
    ks = -(-K // sf_group_k)
    _check_sf(sf_a, "sf_a", G, ks, M_max)
    _check_sf(sf_b, "sf_b", G, ks, N)
    if D is None:
        D = torch.empty((G, M_max, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 3)
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_grouped_masked_blockscaled(
            A.data_ptr(), B.data_ptr(), D.data_ptr(), masked_m.data_ptr(), G, M_max, N, K, int(max_m_hint),
            fa, fb, sf_a.data_ptr(), sf_a.shape[2], sf_b.data_ptr(), sf_b.shape[2], int(sf_group_k),
            int(flags), _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_grouped_masked_blockscaled")
    return D


ACT_NONE, ACT_RELU = 0, 1
ROUND_RN, ROUND_RZ, ROUND_RU, ROUND_RD = 0, 1, 2, 3


def _ex_structs(groups, rows, N, K, scale_a, scale_b, sf_a, sf_b, sf_group_k, epilogue, d_rows=None):
    import torch
    d_rows = groups * rows if d_rows is None else d_rows      # output rows in all
    sc = None
    if scale_a is not None or scale_b is not None or sf_a is not None or sf_b is not None:
        sc = _lib.Scales()
        if scale_a is not None or scale_b is not None:
            if scale_a is None or scale_b is None:
                raise ValueError("output scales need both scale_a and scale_b")
            _check_scale(scale_a, "scale_a", (groups, d_rows))
            _check_scale(scale_b, "scale_b", (groups, groups * N))
            sc.out_a, sc.out_a_len = scale_a.data_ptr(), scale_a.numel()
            sc.out_b, sc.out_b_len = scale_b.data_ptr(), scale_b.numel()
        if sf_a is not None or sf_b is not None:
            if sf_a is None or sf_b is None:
                raise ValueError("block scales need both sf_a and sf_b")
            if sf_group_k not in (32, 128):
                raise ValueError("sf_group_k must be 32 or 128")
            ks = -(-K // sf_group_k)
            sa = sf_a if sf_a.dim() == 3 else sf_a.unsqueeze(0)
            sb = sf_b if sf_b.dim() == 3 else sf_b.unsqueeze(0)
            _check_sf(sa, "sf_a", groups, ks, rows)
            _check_sf(sb, "sf_b", groups, ks, N)
            sc.block_a, sc.block_a_ld = sa.data_ptr(), sa.shape[2]
            sc.block_b, sc.block_b_ld = sb.data_ptr(), sb.shape[2]
            sc.block_k = int(sf_group_k)
    ep = None
    if epilogue is not None:
        e = dict(epilogue)
        ep = _lib.Epilogue()
        ep.alpha = float(e.get("alpha", 1.0))
        ep.beta = float(e.get("beta", 0.0))
        C, bias = e.get("C"), e.get("bias")
        if C is not None:
            if not C.is_cuda or C.dtype != torch.bfloat16 or not C.is_contiguous() or C.numel() != d_rows * N:
                raise ValueError("epilogue C must be a contiguous bf16 CUDA tensor shaped like D")
            ep.c = C.data_ptr()
        if bias is not None:
            if not bias.is_cuda or bias.dtype != torch.float32 or not bias.is_contiguous() or bias.numel() != groups * N:
                raise ValueError("epilogue bias must be a contiguous float32 CUDA tensor of %d entries" % (groups * N))
            ep.bias = bias.data_ptr()
        ep.activation = ACT_RELU if e.get("relu", False) else ACT_NONE
        ep.round_mode = int(e.get("round_mode", ROUND_RN))
    return sc, ep


def fp8_gemm_nt_ex(A, B, D=None, scale_a=None, scale_b=None, sf_a=None, sf_b=None, sf_group_k: int = 128,
                   epilogue=None, a_dtype=None, b_dtype=None, flags: int = 0, stream=None):
    """General dense form: optional output scales (scale_a/scale_b), block
    scales (sf_a/sf_b, sf_group_k) and a fused epilogue given as a dict with
    keys alpha, beta, C (bf16 like D), bias (float32 [N]), relu, round_mode:
    D = round(act(alpha * value + beta * C + bias))."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 2)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M, K = A.shape
    N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch: A has %d, B has %d" % (K, K2))
    sc, ep = _ex_structs(1, M, N, K, scale_a, scale_b, sf_a, sf_b, sf_group_k, epilogue)
    if D is None:
        D = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 2)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (M, N):
            raise ValueError("D must be a contiguous bf16 [M, N] tensor")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_nt_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, fa, fb,
                                        None if sc is None else ctypes.byref(sc),
                                        None if ep is None else ctypes.byref(ep), int(flags),
                                        _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_nt_ex")
    return D


def fp8_gemm_grouped_masked_ex(A, B, masked_m, D=None, max_m_hint: int = 0, scale_a=None, scale_b=None,
                               sf_a=None, sf_b=None, sf_group_k: int = 128, epilogue=None, a_dtype=None,
                               b_dtype=None, flags: int = 0, stream=None):
    """General masked grouped form (see fp8_gemm_nt_ex); epilogue bias is
    float32 [G, N], C bf16 [G, M_max, N]."""
    import torch
    _check_operand(A, "A", 3)
    _check_operand(B, "B", 3)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    G, M_max, K = A.shape
    G2, N, K2 = B.shape
    if G != G2 or K != K2:
        raise ValueError("shape mismatch: A %s, B %s" % (tuple(A.shape), tuple(B.shape)))
    if not masked_m.is_cuda or masked_m.dtype != torch.int32 or tuple(masked_m.shape) != (G,):
        raise ValueError("masked_m must be a contiguous int32 CUDA tensor of shape [G]")
    sc, ep = _ex_structs(G, M_max, N, K, scale_a, scale_b, sf_a, sf_b, sf_group_k, epilogue)
    if D is None:
        D = torch.empty((G, M_max, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 3)
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_grouped_masked_ex(
            A.data_ptr(), B.data_ptr(), D.data_ptr(), masked_m.data_ptr(), G, M_max, N, K, int(max_m_hint), fa, fb,
            None if sc is None else ctypes.byref(sc), None if ep is None else ctypes.byref(ep), int(flags),
            _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_grouped_masked_ex")
    return D


def fp8_gemm_grouped_contiguous(A, B, group_offsets, D=None, max_m_hint: int = 0, scale_a=None, scale_b=None,
                                epilogue=None, a_dtype=None, b_dtype=None, flags: int = 0, stream=None):
    """Contiguous grouped GEMM: A [M_total, K] holds the groups' token rows
    back to back, group g owning rows group_offsets[g] .. group_offsets[g+1]-1
    (int32 CUDA tensor [G+1]); B [G, N, K]; D [M_total, N] (rows outside every
    group untouched).  Optional output scales (scale_a: G or M_total entries,
    scale_b: G or G*N) and fused epilogue (bias [G, N], C like D)."""
    import torch
    _check_operand(A, "A", 2)
    _check_operand(B, "B", 3)
    fa, fb = _fp8_code(A, a_dtype), _fp8_code(B, b_dtype)
    M_total, K = A.shape
    G, N, K2 = B.shape
    if K != K2:
        raise ValueError("K mismatch: A has %d, B has %d" % (K, K2))
    off = group_offsets
    if not off.is_cuda or off.dtype != torch.int32 or not off.is_contiguous() or tuple(off.shape) != (G + 1,):
        raise ValueError("group_offsets must be a contiguous int32 CUDA tensor of shape [G + 1]")
    sc, ep = _ex_structs(G, M_total, N, K, scale_a, scale_b, None, None, 128, epilogue, d_rows=M_total)
    if D is None:
        D = torch.empty((M_total, N), dtype=torch.bfloat16, device=A.device)
    else:
        _check_operand(D, "D", 2)
        if D.dtype != torch.bfloat16 or tuple(D.shape) != (M_total, N):
            raise ValueError("D must be a contiguous bf16 [M_total, N] tensor")
    with _on_device(A.device):
        rc = _lib.load().fp8_gemm_grouped_contiguous_ex(
            A.data_ptr(), B.data_ptr(), D.data_ptr(), off.data_ptr(), G, M_total, N, K, int(max_m_hint), fa, fb,
            None if sc is None else ctypes.byref(sc), None if ep is None else ctypes.byref(ep), int(flags),
            _stream_handle(stream))
    if rc != OK:
        raise Fp8gError(rc, "fp8_gemm_grouped_contiguous")
    return D
