"""GPU parity of the contiguous grouped layout (groups' token rows concatenated
along M, boundaries from device group offsets) against the oracle: unaligned
and empty groups, rows outside every group left untouched, every kernel
path, output scales and the fused epilogue, the same problem in the masked
layout, and offsets that break the rules.  Sources: "一次“转置”，半张算力：
DeepSeek SwapAB 漂流史" §3.1 (grouped GEMM for MoE) and §5 (several grouped
layouts on SM100)."""
import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
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


def run_case(sizes, N, K, flags, hint, seed, lead=3, tail=5, fa=E4, fb=E4, expect_status=fp8g.OK):
    G = len(sizes)
    off = np.concatenate([[lead], lead + np.cumsum(sizes)]).astype(np.int32)
    M_total = int(off[-1]) + tail
    A = synth.normal_fp8((M_total, K), seed, 0.0, 1.0, fa)
    B = synth.normal_fp8((G, N, K), seed + 1, 0.0, 0.5, fb)
    D0 = synth.u16_pattern((M_total, N), seed + 2)
    D0[:, ::53] = 0x7FC2
    Dt = as_bf16(D0)
    fp8g.fp8_gemm_grouped_contiguous(dev(A), dev(B), dev(off), D=Dt, max_m_hint=hint, a_dtype=fa, b_dtype=fb,
                                     flags=flags)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == expect_status, st
    got = bits(Dt)
    ref, absdot = oracle.gemm_grouped_contiguous(A, B, off, D0, fa, fb)
    inside = np.zeros(M_total, bool)
    for g in range(G):
        inside[off[g]:off[g + 1]] = True
    ok, rep = oracle.check_bf16(got[inside], ref[inside], absdot[inside])
    assert ok, rep
    assert np.array_equal(got[~inside], D0[~inside]), "rows outside every group written"
    return got


SIZES = [0, 1, 17, 130, 5, 0, 64, 300, 33]


@pytest.mark.parametrize("flags,hint", [(OFF, 0), (ON, 0), (ON | fp8g.WHOLE_TILES, 0), (AUTO, 0), (AUTO, 48),
                                        (ON, 48)])
def test_unaligned_groups(flags, hint):
    run_case(SIZES, 384, 1024, flags, hint, seed=900)


@pytest.mark.parametrize("flags", [OFF, ON])
def test_many_small_groups_e5m2(flags):
    sizes = list(np.random.default_rng(901).integers(0, 24, 40))
    run_case(sizes, 256, 512, flags, 24, seed=902, fb=E5)


@pytest.mark.parametrize("flags", [OFF, OFF | fp8g.PAIR_TILES, OFF | fp8g.SINGLE_SM_TILES])
def test_large_groups_pair_tiles(flags):
    # about 377 tokens per group on average: SM-pair tiles by default
    run_case([700, 0, 256, 1000, 1, 300], 512, 768, flags, 0, seed=920)


def test_single_group_is_dense():
    run_case([700], 512, 768, OFF, 0, seed=903, lead=0, tail=0)


def test_matches_masked_layout():
    G, M_max, N, K = 6, 64, 256, 640
    mm = np.array([5, 64, 0, 31, 17, 2], np.int32)
    A = synth.normal_fp8((G, M_max, K), 904, 0.0, 1.0, E4)
    B = synth.normal_fp8((G, N, K), 905, 0.0, 0.5, E4)
    Dm = fp8g.fp8_gemm_grouped_masked(dev(A), dev(B), dev(mm), max_m_hint=64, a_dtype=E4, b_dtype=E4, flags=ON)
    off = np.concatenate([[0], np.cumsum(mm)]).astype(np.int32)
    Ac = np.concatenate([A[g, :mm[g]] for g in range(G)])
    for flags in (ON, OFF):
        Dc = fp8g.fp8_gemm_grouped_contiguous(dev(Ac), dev(B), dev(off), max_m_hint=64, a_dtype=E4, b_dtype=E4,
                                              flags=flags)
        torch.cuda.synchronize()
        assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
        want = np.concatenate([bits(Dm)[g, :mm[g]] for g in range(G)])
        if flags == ON:
            assert np.array_equal(bits(Dc), want)        # same kernel, same arithmetic
        else:
            ref, absdot = oracle.gemm_grouped_contiguous(Ac, B, off)
            ok, rep = oracle.check_bf16(bits(Dc), ref, absdot)
            assert ok, rep


@pytest.mark.parametrize("flags,sizes", [(OFF, [40, 0, 129, 7]), (ON, [40, 0, 129, 7]),
                                         (OFF | fp8g.PAIR_TILES, [300, 0, 520, 7])])
def test_scales_and_epilogue(flags, sizes):
    G, N, K = len(sizes), 256, 512
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    M_total = int(off[-1])
    A = synth.normal_fp8((M_total, K), 906, 0.0, 1.0, E4)
    B = synth.normal_fp8((G, N, K), 907, 0.0, 0.5, E4)
    rng = np.random.default_rng(908)
    sa = np.exp2(rng.uniform(-4, 4, M_total)).astype(np.float32)         # per row
    sb = np.exp2(rng.uniform(-4, 4, G * N)).astype(np.float32)           # per group and column
    bias = rng.standard_normal((G, N)).astype(np.float32)
    C = oracle.round_bf16_array(rng.standard_normal((M_total, N)))
    D = fp8g.fp8_gemm_grouped_contiguous(dev(A), dev(B), dev(off), scale_a=dev(sa), scale_b=dev(sb),
                                         epilogue={"alpha": 2.0, "beta": -1.0, "C": as_bf16(C), "bias": dev(bias),
                                                   "relu": True},
                                         a_dtype=E4, b_dtype=E4, flags=flags)
    torch.cuda.synchronize()
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
    _, absS, S = oracle.gemm_grouped_contiguous(A, B, off, want_exact=True)
    gid = np.repeat(np.arange(G), sizes)
    f = sa.astype(np.float64)[:, None] * sb.reshape(G, N).astype(np.float64)[gid]
    # one "group" per row for the oracle, so that each row sees its group's bias
    ref, absdot = oracle.epilogue((S * f).reshape(M_total, 1, N), (absS * np.abs(f)).reshape(M_total, 1, N), 2.0,
                                  -1.0, C.reshape(M_total, 1, N), bias[gid], True, 0)
    ok, rep = oracle.check_bf16(bits(D), ref.reshape(M_total, N), absdot.reshape(M_total, N))
    assert ok, rep


def test_bad_offsets_skip_the_group_and_report():
    """Group 1 claims rows past M_total: it is skipped and reported; the
    other groups are still computed."""
    G, N, K = 3, 128, 256
    M_total = 50
    off = np.array([0, 20, 70, 50], np.int32)       # group 1 ends past M_total, group 2 is reversed
    A = synth.normal_fp8((M_total, K), 909, 0.0, 1.0, E4)
    B = synth.normal_fp8((G, N, K), 910, 0.0, 0.5, E4)
    D0 = synth.u16_pattern((M_total, N), 911)
    Dt = as_bf16(D0)
    fp8g.fp8_gemm_grouped_contiguous(dev(A), dev(B), dev(off), D=Dt, a_dtype=E4, b_dtype=E4, flags=OFF)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.ERR_MASKED_M_RANGE, st
    got = bits(Dt)
    ref, absdot = oracle.gemm_nt(A[:20], B[0])
    ok, rep = oracle.check_bf16(got[:20], ref, absdot)
    assert ok, rep
    assert np.array_equal(got[20:], D0[20:])


def test_block_scales_rejected():
    A = torch.zeros((64, 128), dtype=torch.uint8, device="cuda")
    B = torch.zeros((2, 64, 128), dtype=torch.uint8, device="cuda")
    off = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    sf = torch.full((1, 1, 64), 127, dtype=torch.uint8, device="cuda")
    sc = fp8g._lib.Scales()
    sc.block_a, sc.block_a_ld, sc.block_b, sc.block_b_ld, sc.block_k = sf.data_ptr(), 64, sf.data_ptr(), 64, 128
    D = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")
    import ctypes
    rc = fp8g._lib.load().fp8_gemm_grouped_contiguous_ex(A.data_ptr(), B.data_ptr(), D.data_ptr(), off.data_ptr(), 2,
                                                         64, 64, 128, 0, 0, 0, ctypes.byref(sc), None, 0, None)
    assert rc == fp8g.ERR_UNSUPPORTED
