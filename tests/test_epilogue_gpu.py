"""GPU parity of the fused epilogue (alpha * value + beta * C + bias, ReLU,
BF16 rounding mode) against the oracle's epilogue definition, on every
kernel the dispatcher can choose, combined with output scales and block
scales, in place (C == D), and with masked groups whose padding rows must be
neither read nor written.  Source: "DeepGEMM：基于 Hopper Tensor Core 的 FP8
矩阵乘法内核优化实践" §3.3 (epilogue fusion, rounding modes)."""
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


def as_bf16(codes):
    return dev(np.ascontiguousarray(codes, np.uint16).view(np.int16)).view(torch.bfloat16)


def assert_status_ok():
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, "device status %s" % (st,)


def c_codes(shape, seed):
    """BF16 codes of moderate magnitude, both signs."""
    v = np.random.default_rng(seed).standard_normal(shape) * 4.0
    return oracle.round_bf16_array(v)


KERNELS = {"pair": OFF, "pair_stream_k": OFF | fp8g.STREAM_K, "single_sm": OFF | fp8g.SINGLE_SM_TILES,
           "swap_stream_k": ON, "swap_whole": ON | fp8g.WHOLE_TILES}


def run_dense(M, N, K, kernel, alpha, beta, use_c, use_bias, relu, mode, seed, in_place=False):
    A = synth.normal_fp8((M, K), seed, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), seed + 1, 0.0, 1.0, E4)
    C = c_codes((M, N), seed + 2) if use_c else None
    bias = (np.random.default_rng(seed + 3).standard_normal(N) * 8).astype(np.float32) if use_bias else None
    epi = {"alpha": alpha, "beta": beta, "relu": relu, "round_mode": mode}
    Ct = as_bf16(C) if use_c else None
    if use_c:
        epi["C"] = Ct
    if use_bias:
        epi["bias"] = dev(bias)
    D = Ct if in_place else None
    out = fp8g.fp8_gemm_nt_ex(dev(A), dev(B), D=D, epilogue=epi, a_dtype=E4, b_dtype=E4, flags=KERNELS[kernel])
    torch.cuda.synchronize()
    assert_status_ok()
    _, absS, S = oracle.gemm_nt(A, B, want_exact=True)
    ref, absdot = oracle.epilogue(S, absS, alpha, beta, C, bias, relu, mode)
    ok, rep = oracle.check_bf16(bits(out), ref, absdot)
    assert ok, rep


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_dense_full_epilogue(kernel, mode):
    M, N, K = (40, 640, 1536) if kernel.startswith("swap") else (392, 544, 640)
    run_dense(M, N, K, kernel, 0.75, -1.5, True, True, mode == 1, mode,
              seed=700 + 10 * sorted(KERNELS).index(kernel) + mode)


@pytest.mark.parametrize("kernel", ["pair", "single_sm", "swap_stream_k"])
def test_dense_in_place_accumulate(kernel):
    """D = AB + D: C and D are the same buffer."""
    M, N, K = (48, 384, 1024) if kernel.startswith("swap") else (300, 256, 512)
    run_dense(M, N, K, kernel, 1.0, 1.0, True, False, False, 0, seed=760, in_place=True)


@pytest.mark.parametrize("kernel", ["pair", "swap_whole"])
def test_dense_bias_relu_only(kernel):
    M, N, K = (16, 512, 768) if kernel.startswith("swap") else (256, 512, 768)
    run_dense(M, N, K, kernel, 1.0, 0.0, False, True, True, 0, seed=770)


def test_epilogue_with_output_and_block_scales():
    M, N, K = 260, 384, 640
    A = synth.normal_fp8((M, K), 780, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 781, 0.0, 1.0, E4)
    rng = np.random.default_rng(782)
    ks = K // 128
    sfa = rng.integers(120, 135, (ks, 272)).astype(np.uint8)
    sfb = rng.integers(120, 135, (ks, N)).astype(np.uint8)
    sa = np.exp2(rng.uniform(-3, 3, M)).astype(np.float32)
    sb = np.exp2(rng.uniform(-3, 3, N)).astype(np.float32)
    C = c_codes((M, N), 783)
    bias = rng.standard_normal(N).astype(np.float32)
    for flags in (OFF, ON):
        out = fp8g.fp8_gemm_nt_ex(dev(A), dev(B), scale_a=dev(sa), scale_b=dev(sb), sf_a=dev(sfa), sf_b=dev(sfb),
                                  epilogue={"alpha": 0.5, "beta": 2.0, "C": as_bf16(C), "bias": dev(bias),
                                            "relu": True, "round_mode": 2},
                                  a_dtype=E4, b_dtype=E4, flags=flags)
        torch.cuda.synchronize()
        assert_status_ok()
        _, absS, S = oracle.gemm_blockscaled(A, B, sfa, sfb, 128, want_exact=True)
        f = sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
        ref, absdot = oracle.epilogue(S * f, absS * np.abs(f), 0.5, 2.0, C, bias, True, 2)
        ok, rep = oracle.check_bf16(bits(out), ref, absdot)
        assert ok, (flags, rep)


@pytest.mark.parametrize("flags,hint", [(ON, 32), (ON | fp8g.WHOLE_TILES, 64), (OFF, 0)])
def test_grouped_epilogue_padding_neither_read_nor_written(flags, hint):
    G, M_max, N, K = 6, 64, 384, 512
    A = synth.normal_fp8((G, M_max, K), 790, 0.0, 0.5, E4)
    B = synth.normal_fp8((G, N, K), 791, 0.0, 0.5, E4)
    mm = np.array([0, 1, 17, 64, 33, 8], np.int32)
    C = c_codes((G, M_max, N), 792)
    D0 = synth.u16_pattern((G, M_max, N), 793)
    for g in range(G):
        C[g, mm[g]:] = 0x7FC0                   # NaN in C's padding rows: never read
    bias = np.random.default_rng(794).standard_normal((G, N)).astype(np.float32)
    Dt = as_bf16(D0)
    fp8g.fp8_gemm_grouped_masked_ex(dev(A), dev(B), dev(mm), D=Dt, max_m_hint=hint,
                                    epilogue={"alpha": -1.0, "beta": 0.5, "C": as_bf16(C), "bias": dev(bias),
                                              "round_mode": 1},
                                    a_dtype=E4, b_dtype=E4, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    got = bits(Dt)
    S = np.zeros((G, M_max, N))
    absS = np.zeros((G, M_max, N))
    for g in range(G):
        if mm[g]:
            _, a_, s_ = oracle.gemm_nt(A[g, :mm[g]], B[g], want_exact=True)
            S[g, :mm[g]], absS[g, :mm[g]] = s_, a_
    ref, absdot = oracle.epilogue(S, absS, -1.0, 0.5, C, bias, False, 1, masked_m=mm, D_init=D0)
    for g in range(G):
        m = mm[g]
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:])


def test_grouped_epilogue_with_block_scales():
    G, M_max, N, K = 4, 32, 256, 640
    A = synth.normal_fp8((G, M_max, K), 800, 0.0, 0.5, E4)
    B = synth.normal_fp8((G, N, K), 801, 0.0, 0.5, E4)
    mm = np.array([32, 3, 0, 20], np.int32)
    rng = np.random.default_rng(802)
    ks = K // 32
    sfa = rng.integers(120, 135, (G, ks, M_max)).astype(np.uint8)
    sfb = rng.integers(120, 135, (G, ks, N)).astype(np.uint8)
    bias = rng.standard_normal((G, N)).astype(np.float32)
    D0 = synth.u16_pattern((G, M_max, N), 803)
    Dt = as_bf16(D0)
    fp8g.fp8_gemm_grouped_masked_ex(dev(A), dev(B), dev(mm), D=Dt, max_m_hint=32, sf_a=dev(sfa), sf_b=dev(sfb),
                                    sf_group_k=32, epilogue={"bias": dev(bias), "relu": True},
                                    a_dtype=E4, b_dtype=E4, flags=AUTO)
    torch.cuda.synchronize()
    assert_status_ok()
    _, absS, S = oracle.gemm_blockscaled(A, B, sfa, sfb, 32, masked_m=mm, D_init=D0, want_exact=True)
    ref, absdot = oracle.epilogue(S, absS, 1.0, 0.0, None, bias, True, 0, masked_m=mm, D_init=D0)
    got = bits(Dt)
    for g in range(G):
        m = mm[g]
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:])


def test_epilogue_argument_errors():
    lib = _lib.load()
    A = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    B = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    D = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(80, dtype=torch.float32, device="cuda")

    def call(**kw):
        e = _lib.Epilogue()
        e.alpha, e.beta = 1.0, 0.0
        for k, v in kw.items():
            setattr(e, k, v)
        return lib.fp8_gemm_nt_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), 64, 64, 128, 0, 0, None,
                                  ctypes.byref(e), 0, None)
    assert call() == fp8g.OK
    assert call(activation=2) == fp8g.ERR_INVALID_ARG
    assert call(round_mode=4) == fp8g.ERR_INVALID_ARG
    assert call(round_mode=-1) == fp8g.ERR_INVALID_ARG
    assert call(bias=bias.data_ptr() + 4) == fp8g.ERR_MISALIGNED
    assert call(c=D.data_ptr() + 2) == fp8g.ERR_MISALIGNED
    sc = _lib.Scales()
    sc.out_a = bias.data_ptr()
    sc.out_a_len = 1
    assert lib.fp8_gemm_nt_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), 64, 64, 128, 0, 0, ctypes.byref(sc), None,
                              0, None) == fp8g.ERR_INVALID_ARG        # out_b missing
    torch.cuda.synchronize()
    assert_status_ok()
