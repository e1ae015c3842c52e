"""GPU parity of the scaled entry points (output multiplied by per-tensor or
per-channel FP32 scales before the BF16 rounding, as in "DeepGEMM：基于
Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §3.1 and §5.2) against the
oracle's scaled definition, on every kernel the dispatcher can choose, and
the host-side argument checks."""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
from fp8_tensor_core_gb300 import _lib
import oracle
import synth

pytestmark = pytest.mark.gpu

E4, E5 = synth.E4M3, synth.E5M2
OFF, ON, AUTO = fp8g.SWAP_OFF, fp8g.SWAP_ON, fp8g.SWAP_AUTO


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()
    torch.cuda.set_device(0)
    fp8g.fp8g_get_device_status()
    yield


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_status_ok():
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, "device status %s" % (st,)


def scales(n, seed, spread=6.0, negative=True):
    """Seeded FP32 scales 2^u, u uniform in [-spread, spread], some negated."""
    rng = np.random.default_rng(seed)
    s = np.exp2(rng.uniform(-spread, spread, n))
    if negative:
        s *= np.where(rng.random(n) < 0.25, -1.0, 1.0)
    return s.astype(np.float32)


def check_dense_scaled(M, N, K, sa_len, sb_len, flags, seed, fa=E4, fb=E4):
    A = synth.normal_fp8((M, K), seed, 0.0, 1.0, fa)
    B = synth.normal_fp8((N, K), seed + 1, 0.0, 1.0, fb)
    sa = scales(sa_len, seed + 2)
    sb = scales(sb_len, seed + 3)
    D = fp8g.fp8_gemm_nt_scaled(dev(A), dev(B), dev(sa), dev(sb), a_dtype=fa, b_dtype=fb, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    ref, absdot = oracle.gemm_nt_scaled(A, B, sa, sb, fa, fb)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot)
    assert ok, rep
    return rep


KERNELS = {
    "pair": OFF,
    "pair_stream_k": OFF | fp8g.STREAM_K,
    "single_sm": OFF | fp8g.SINGLE_SM_TILES,
    "swap_stream_k": ON,
    "swap_whole": ON | fp8g.WHOLE_TILES,
    "swap_share_sm": ON | fp8g.SHARE_SM,
}


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("per_row,per_col", [(False, False), (True, True), (True, False), (False, True)])
def test_dense_scaled_every_kernel(kernel, per_row, per_col):
    M, N, K = (48, 640, 1536) if kernel.startswith("swap") else (392, 544, 640)
    check_dense_scaled(M, N, K, M if per_row else 1, N if per_col else 1, KERNELS[kernel],
                       seed=300 + 7 * sorted(KERNELS).index(kernel) + 2 * per_row + per_col)


@pytest.mark.parametrize("fa,fb", [(E5, E4), (E4, E5), (E5, E5)])
def test_dense_scaled_mixed_formats(fa, fb):
    check_dense_scaled(200, 272, 384, 200, 272, AUTO, seed=340, fa=fa, fb=fb)


@pytest.mark.parametrize("M", [1, 16, 33])
def test_dense_scaled_small_m_auto(M):
    check_dense_scaled(M, 2048, 1024, M, 2048, AUTO, seed=350 + M)


def test_unit_scales_match_unscaled_bitwise():
    A = synth.normal_fp8((300, 512), 360, 0.0, 1.0, E4)
    B = synth.normal_fp8((400, 512), 361, 0.0, 1.0, E4)
    for flags in (OFF, ON, OFF | fp8g.SINGLE_SM_TILES):
        D0 = fp8g.fp8_gemm_nt(dev(A), dev(B), a_dtype=E4, b_dtype=E4, flags=flags)
        D1 = fp8g.fp8_gemm_nt_scaled(dev(A), dev(B), dev(np.ones(300, np.float32)),
                                     dev(np.ones(1, np.float32)), a_dtype=E4, b_dtype=E4, flags=flags)
        torch.cuda.synchronize()
        assert_status_ok()
        assert np.array_equal(bits(D0), bits(D1)), flags


def test_power_of_two_scales_shift_exponents_exactly():
    """Integer data whose sums are exact in FP32 and BF16: scaling by 2^e
    shifts the exponent of every (bit-exact) unscaled result."""
    M, N, K = 256, 256, 256
    A = synth.uniform_fp8((M, K), 370, -2.0, 2.0, E4)
    B = synth.uniform_fp8((N, K), 371, -2.0, 2.0, E4)
    rng = np.random.default_rng(372)
    ea = rng.integers(-20, 21, M)
    eb = rng.integers(-20, 21, N)
    sa = np.ldexp(1.0, ea).astype(np.float32)
    sb = np.ldexp(1.0, eb).astype(np.float32)
    for flags in (OFF, ON, OFF | fp8g.SINGLE_SM_TILES):
        D0 = bits(fp8g.fp8_gemm_nt(dev(A), dev(B), a_dtype=E4, b_dtype=E4, flags=flags))
        D1 = bits(fp8g.fp8_gemm_nt_scaled(dev(A), dev(B), dev(sa), dev(sb), a_dtype=E4, b_dtype=E4,
                                          flags=flags))
        torch.cuda.synchronize()
        assert_status_ok()
        want = oracle.bf16_bits_to_f64(D0) * np.ldexp(1.0, ea[:, None] + eb[None, :])
        assert np.array_equal(oracle.bf16_bits_to_f64(D1), want), flags


# ---- grouped ----------------------------------------------------------------------

def grouped_scaled_case(G, M_max, N, K, mm, sa_per_row, sb_per_col, flags, hint, seed):
    A = synth.normal_fp8((G, M_max, K), seed, 0.0, 0.5, E4)
    B = synth.normal_fp8((G, N, K), seed + 1, 0.0, 0.5, E4)
    mm = np.asarray(mm, np.int32)
    sa = scales(G * M_max if sa_per_row else G, seed + 2)
    sb = scales(G * N if sb_per_col else G, seed + 3)
    D0 = synth.u16_pattern((G, M_max, N), seed + 4)
    D0[..., ::89] = 0x7FC1
    Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked_scaled(dev(A), dev(B), dev(mm), dev(sa), dev(sb), D=Dt,
                                        max_m_hint=hint, a_dtype=E4, b_dtype=E4, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    got = bits(Dt)
    ref, absdot = oracle.gemm_grouped_masked_scaled(A, B, mm, sa, sb, D0, E4, E4)
    for g in range(G):
        m = mm[g]
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g


@pytest.mark.parametrize("flags,hint", [(ON, 32), (ON | fp8g.WHOLE_TILES, 32), (OFF, 0), (AUTO, 0)])
@pytest.mark.parametrize("sa_per_row,sb_per_col", [(False, False), (True, True), (False, True)])
def test_grouped_scaled(flags, hint, sa_per_row, sb_per_col):
    mm = [0, 1, 9, 16, 17, 32, 5, 64]
    grouped_scaled_case(len(mm), 64, 384, 512, mm, sa_per_row, sb_per_col, flags, hint,
                        seed=400 + 4 * sa_per_row + 2 * sb_per_col)


def test_grouped_scaled_moe_decode_shape():
    """The MoE-decode shape (weights 4096 x 7168 per expert) with per-token
    and per-channel scales, sampled groups."""
    G, M_max, N, K = 8, 64, 4096, 7168
    mm = [3, 64, 0, 17, 40, 1, 8, 33]
    grouped_scaled_case(G, M_max, N, K, mm, True, True, AUTO, 64, seed=420)


# ---- host-side argument checks (no kernel runs) -------------------------------------

def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_scaled_argument_errors():
    lib = _lib.load()
    A = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    D = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.ones(80, dtype=torch.float32, device="cuda")
    def call(sa, sa_len, sb, sb_len):
        return lib.fp8_gemm_nt_scaled(_ptr(A), _ptr(B), _ptr(D), 64, 64, 128, 0, 0, sa, sa_len, sb, sb_len,
                                      0, None)
    assert call(_ptr(s), 1, _ptr(s), 1) == fp8g.OK
    assert call(_ptr(s), 64, _ptr(s), 64) == fp8g.OK
    assert call(None, 1, _ptr(s), 1) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 1, None, 1) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 2, _ptr(s), 1) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 1, _ptr(s), 65) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 0, _ptr(s), 1) == fp8g.ERR_INVALID_ARG
    off = ctypes.c_void_p(s.data_ptr() + 4)
    assert call(off, 1, _ptr(s), 1) == fp8g.ERR_MISALIGNED
    assert call(_ptr(s), 1, off, 1) == fp8g.ERR_MISALIGNED
    mm = torch.zeros(2, dtype=torch.int32, device="cuda")
    A3 = torch.zeros((2, 32, 128), dtype=torch.uint8, device="cuda")
    B3 = torch.zeros((2, 32, 128), dtype=torch.uint8, device="cuda")
    D3 = torch.zeros((2, 32, 32), dtype=torch.bfloat16, device="cuda")
    def gcall(sa_len, sb_len):
        return lib.fp8_gemm_grouped_masked_scaled(_ptr(A3), _ptr(B3), _ptr(D3), _ptr(mm), 2, 32, 32, 128, 0,
                                                  0, 0, _ptr(s), sa_len, _ptr(s), sb_len, 0, None)
    assert gcall(2, 2) == fp8g.OK
    assert gcall(64, 64) == fp8g.OK
    assert gcall(1, 2) == fp8g.ERR_INVALID_ARG
    assert gcall(2, 32) == fp8g.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert_status_ok()
    with pytest.raises(ValueError):
        fp8g.fp8_gemm_nt_scaled(A, B, s[:3], s[:1], a_dtype=E4, b_dtype=E4)
    with pytest.raises(ValueError):
        fp8g.fp8_gemm_nt_scaled(A, B, s[:1].double(), s[:1], a_dtype=E4, b_dtype=E4)
