"""SM-pair tiles with the last partial wave split along K.

When the tiles left after the whole waves of 256-row SM-pair tiles number at
most half the pairs, each of them can be split s ways along K ("DeepGEMM：基于
Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §1.3: every SM busy on large
shapes), run before the pairs' whole tiles; the last contributor of a tile
sums the others' FP32 partial tiles with its own in K order (§6.4: a fixed
order, no unordered atomic accumulation).  Shapes here are chosen so that
the planner (pinned through fp8g_describe_plan for this device) picks s = 2,
3 and 4, with ranges that straddle tiles, ragged M, N and K, with and
without whole waves; every element is checked against the oracle on two
calls in a row (the arrival counters must be back at zero after a launch)."""
import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
import oracle
import synth

pytestmark = pytest.mark.gpu

E4, E5 = synth.E4M3, synth.E5M2


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()
    torch.cuda.set_device(0)
    fp8g.fp8g_get_device_status()
    yield


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def plan_of(M, N, K, sf=0, flags=0):
    props = torch.cuda.get_device_properties(0)
    if props.multi_processor_count != 152:
        pytest.skip("split choices are pinned for 152 SMs")
    return fp8g.fp8g_describe_plan(fp8g.LAYOUT_DENSE, 1, M, N, K, 0, sf, flags)


# (M, N, K, B format, flags, expected split).  By default the split needs a
# whole wave of tiles besides (4096 x 4096 x 3072, 4000 x 4088 x 4096);
# FP8G_SPLIT_TAIL forces it: without whole waves (s = 2, 3, 4; 128- and
# 160-wide tiles), ranges that straddle tiles (s = 3 over 64 and 32 K blocks),
# ragged M, N and K, and whole waves plus a split tail at short K.
SPLIT = fp8g.SPLIT_TAIL
CASES = [(4096, 4096, 3072, E4, 0, 2), (4000, 4088, 4096, E4, 0, 2), (1000, 1016, 4000, E4, SPLIT, 2),
         (1280, 1024, 4096, E4, SPLIT, 2), (512, 1536, 8192, E5, SPLIT, 3), (1024, 4608, 4096, E4, SPLIT, 3),
         (768, 768, 8192, E5, SPLIT, 4), (6400, 2560, 2048, E4, SPLIT, 2)]


@pytest.mark.parametrize("M,N,K,fb,flags,split", CASES)
def test_split_tail_every_element_twice(M, N, K, fb, flags, split):
    plan = plan_of(M, N, K, flags=flags)
    assert plan["kernel"] == fp8g.KERNEL_SM_PAIRS and plan["k_split"] == split, plan
    A = synth.normal_fp8((M, K), 901 + M, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 902 + N, 0.0, 1.0, fb)
    Ad, Bd = dev(A), dev(B)
    ref, absdot = oracle.gemm_nt(A, B, E4, fb)
    first = None
    for call in range(2):
        D = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        st = fp8g.fp8g_get_device_status()
        assert st[0] == fp8g.OK, st
        got = bits(D)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, (call, rep)
        if first is None:
            first = got
        else:
            assert np.array_equal(first, got), "split-tail results differ between calls"


def test_split_tail_whole_tiles_flag_and_fused_epilogue():
    """FP8G_WHOLE_TILES turns the split off; the fused epilogue (output
    scales, alpha, beta*C, bias, ReLU, directed rounding) runs on split
    tiles too."""
    M, N, K = 1280, 1024, 4096
    assert plan_of(M, N, K, flags=fp8g.SPLIT_TAIL | fp8g.WHOLE_TILES)["k_split"] == 1
    assert plan_of(M, N, K, flags=fp8g.SPLIT_TAIL)["k_split"] == 2
    rng = np.random.default_rng(911)
    A = synth.normal_fp8((M, K), 912, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 913, 0.0, 1.0, E4)
    sa = np.exp2(rng.uniform(-3, 3, M)).astype(np.float32)
    sb = np.exp2(rng.uniform(-3, 3, N)).astype(np.float32)
    C = rng.standard_normal((M, N)).astype(np.float32)
    Ct = torch.from_numpy(C).to(torch.bfloat16).cuda()
    Cb = Ct.view(torch.int16).cpu().numpy().view(np.uint16)
    bias = rng.standard_normal(N).astype(np.float32)
    _, absS, S = oracle.gemm_nt(A, B, want_exact=True)
    f = sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
    ref, absdot = oracle.epilogue(S * f, absS * np.abs(f), 0.5, 2.0, Cb, bias, True, 2)
    for flags in (fp8g.SPLIT_TAIL, fp8g.WHOLE_TILES):
        out = fp8g.fp8_gemm_nt_ex(dev(A), dev(B), scale_a=dev(sa), scale_b=dev(sb),
                                  epilogue={"alpha": 0.5, "beta": 2.0, "C": Ct, "bias": dev(bias), "relu": True,
                                            "round_mode": 2}, a_dtype=E4, b_dtype=E4, flags=flags)
        torch.cuda.synchronize()
        assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
        ok, rep = oracle.check_bf16(bits(out), ref, absdot)
        assert ok, (flags, rep)


def test_split_tail_block_scaled_pair_tiles():
    """Block-scaled SM-pair tiles (FP8G_PAIR_TILES) with a split tail: the
    scale-staging warps follow the same segment order."""
    M, N, K = 1280, 1024, 4096
    flags = fp8g.PAIR_TILES | fp8g.SPLIT_TAIL
    plan = plan_of(M, N, K, sf=128, flags=flags)
    assert plan["kernel"] == fp8g.KERNEL_SM_PAIRS and plan["k_split"] >= 2, plan
    rng = np.random.default_rng(921)
    A = synth.normal_fp8((M, K), 922, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 923, 0.0, 1.0, E4)
    ks = K // 128
    sfa = rng.integers(120, 135, (ks, M)).astype(np.uint8)
    sfb = rng.integers(120, 135, (ks, N)).astype(np.uint8)
    D = fp8g.fp8_gemm_nt_blockscaled(dev(A), dev(B), dev(sfa), dev(sfb), sf_group_k=128, a_dtype=E4, b_dtype=E4,
                                     flags=flags)
    torch.cuda.synchronize()
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
    ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, 128, want_accbound=True)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot, acc_bound=accb)
    assert ok, rep


# FP8G_STREAM_K: the 28 tiles after the whole waves share 896 K blocks over
# the 76 pairs in equal ranges of 11-12, so 12 tiles have three contributors
# and 16 have four (the summing contributor then loads the other three's
# partial tiles at once); 24 of them start inside another pair's range.
# Without whole waves and after one.
@pytest.mark.parametrize("M,N,K", [(512, 3584, 4096), (2048, 3328, 4096)])
def test_stream_k_three_and_four_contributors_twice(M, N, K):
    plan = plan_of(M, N, K, flags=fp8g.STREAM_K)
    assert plan["kernel"] == fp8g.KERNEL_SM_PAIRS and plan["k_split"] == 0, plan
    A = synth.normal_fp8((M, K), 931 + M, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 932 + N, 0.0, 1.0, E4)
    Ad, Bd = dev(A), dev(B)
    ref, absdot = oracle.gemm_nt(A, B, E4, E4)
    first = None
    for call in range(2):
        D = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4, flags=fp8g.STREAM_K)
        torch.cuda.synchronize()
        st = fp8g.fp8g_get_device_status()
        assert st[0] == fp8g.OK, st
        got = bits(D)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, (call, rep)
        if first is None:
            first = got
        else:
            assert np.array_equal(first, got), "stream-K results differ between calls"


def test_stream_k_three_and_four_contributors_integer_exact_and_epilogue():
    """Integer-valued products make every FP32 partial and sum exact, so the
    three- and four-contributor sums must equal the oracle bit for bit; the
    fused epilogue (output scales, alpha, beta*C, bias, ReLU, rounding
    toward zero) runs on the same tiles."""
    M, N, K = 512, 3584, 4096
    assert plan_of(M, N, K, flags=fp8g.STREAM_K)["k_split"] == 0
    rng = np.random.default_rng(941)
    # E4M3 codes of -2..2: every partial sum is an integer below 2^14, exact in FP32
    enc = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    A = np.vectorize(enc.get)(rng.choice([-2, -1, 0, 1, 2], (M, K))).astype(np.uint8)
    B = np.vectorize(enc.get)(rng.choice([-2, -1, 0, 1, 2], (N, K))).astype(np.uint8)
    D = fp8g.fp8_gemm_nt(dev(A), dev(B), a_dtype=E4, b_dtype=E4, flags=fp8g.STREAM_K)
    torch.cuda.synchronize()
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
    ref, absdot = oracle.gemm_nt(A, B, E4, E4)
    assert np.array_equal(bits(D), ref)

    A = synth.normal_fp8((M, K), 942, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 943, 0.0, 1.0, E4)
    sa = np.exp2(rng.uniform(-3, 3, M)).astype(np.float32)
    sb = np.exp2(rng.uniform(-3, 3, N)).astype(np.float32)
    C = rng.standard_normal((M, N)).astype(np.float32)
    Ct = torch.from_numpy(C).to(torch.bfloat16).cuda()
    Cb = Ct.view(torch.int16).cpu().numpy().view(np.uint16)
    bias = rng.standard_normal(N).astype(np.float32)
    _, absS, S = oracle.gemm_nt(A, B, want_exact=True)
    f = sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
    ref, absdot = oracle.epilogue(S * f, absS * np.abs(f), 0.5, 2.0, Cb, bias, True, 1)
    out = fp8g.fp8_gemm_nt_ex(dev(A), dev(B), scale_a=dev(sa), scale_b=dev(sb),
                              epilogue={"alpha": 0.5, "beta": 2.0, "C": Ct, "bias": dev(bias), "relu": True,
                                        "round_mode": 1}, a_dtype=E4, b_dtype=E4, flags=fp8g.STREAM_K)
    torch.cuda.synchronize()
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
    ok, rep = oracle.check_bf16(bits(out), ref, absdot)
    assert ok, rep
