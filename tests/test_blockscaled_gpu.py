"""GPU parity of the block-scaled entry points (UE8M0 scale per row per 32- or
128-element K group, applied by tcgen05.mma kind::mxf8f6f4.block_scale)
against the oracle's block-scaled definition: the SM-pair and single-SM tile
kernels at every tile width, SwapAB (stream-K and whole tiles), the masked grouped form
with poisoned padding, ragged tails, both FP8 formats, and the host-side
argument checks.  Sources: "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法
内核优化实践" §5.2 (per-128-element groups) and "一次“转置”，半张算力：DeepSeek
SwapAB 漂流史" §3.4 (scale factors in the Blackwell MMA)."""
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


def ld16(n):
    return -(-n // 16) * 16


def ue8m0(shape, seed, lo=117, hi=137):
    """Seeded UE8M0 codes in [lo, hi] (2^-10 .. 2^10 by default)."""
    return np.random.default_rng(seed).integers(lo, hi + 1, shape).astype(np.uint8)


def check_dense_bs(M, N, K, gran, flags, seed, fa=E4, fb=E4, pad=16):
    A = synth.normal_fp8((M, K), seed, 0.0, 1.0, fa)
    B = synth.normal_fp8((N, K), seed + 1, 0.0, 1.0, fb)
    ks = -(-K // gran)
    sfa = ue8m0((ks, ld16(M) + pad), seed + 2)
    sfb = ue8m0((ks, ld16(N) + pad), seed + 3)
    D = fp8g.fp8_gemm_nt_blockscaled(dev(A), dev(B), dev(sfa), dev(sfb), sf_group_k=gran, a_dtype=fa,
                                     b_dtype=fb, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, fa=fa, fb=fb, want_accbound=True)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot, acc_bound=accb)
    assert ok, rep
    return rep


# ---- token tiles: SM pairs and single SMs (tokens on M) -------------------------------

DENSE_KERNELS = {"pair": OFF | fp8g.PAIR_TILES, "single_sm": OFF | fp8g.SINGLE_SM_TILES,
                 "single_sm_two_issuers": OFF | fp8g.SINGLE_SM_TILES | fp8g.TWO_MMA_ISSUERS,
                 "pair_two_issuers": OFF | fp8g.PAIR_TILES | fp8g.TWO_MMA_ISSUERS,
                 "pair_stream_k_two_issuers": OFF | fp8g.PAIR_TILES | fp8g.STREAM_K | fp8g.TWO_MMA_ISSUERS,
                 "pair_stream_k": OFF | fp8g.PAIR_TILES | fp8g.STREAM_K, "auto": OFF}


@pytest.mark.parametrize("kernel", sorted(DENSE_KERNELS))
@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (300, 520, 1040), (129, 232, 2064), (640, 896, 512)])
def test_dense_tiles(M, N, K, gran, kernel):
    check_dense_bs(M, N, K, gran, DENSE_KERNELS[kernel], seed=500 + M + N + K + gran)


@pytest.mark.parametrize("kernel", ["pair", "single_sm"])
@pytest.mark.parametrize("tn", [4, 5, 6, 7, 8])
def test_dense_every_tile_width(tn, kernel):
    """FP8G_TILE_N(8): 256-wide single-SM tiles with one accumulator buffer;
    SM pairs clamp it to the widest block-scaled tile."""
    check_dense_bs(256, 480, 768, 128, DENSE_KERNELS[kernel] | fp8g.TILE_N(tn), seed=520 + tn)


@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("M,N,K", [(300, 640, 6272), (129, 520, 8208)])
def test_single_sm_long_k_wide_tiles(M, N, K, gran):
    """K of 49 / 65 K blocks: 256-wide single-SM tiles with one buffer (the
    default from 48 K blocks), N tails inside a tile, several tiles per SM."""
    check_dense_bs(M, N, K, gran, OFF | fp8g.SINGLE_SM_TILES, seed=540 + M + gran)


@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("tn", [1, 2, 3])
def test_single_sm_narrow_tiles_two_issuers(tn, gran):
    """Tiles of 32..96 columns: two MMA issuers with two accumulator buffers each."""
    check_dense_bs(300, 416, 1664, gran, OFF | fp8g.SINGLE_SM_TILES | fp8g.TILE_N(tn), seed=527 + tn + gran)
    check_dense_bs(300, 416, 1664, gran, OFF | fp8g.SINGLE_SM_TILES | fp8g.TILE_N(tn) | fp8g.ONE_MMA_ISSUER,
                   seed=527 + tn + gran)


@pytest.mark.parametrize("stages", [0, 1, 2])
@pytest.mark.parametrize("K", [256, 384, 640])
def test_single_sm_scale_ring_across_tiles(K, stages):
    """128-element groups on single-SM tiles: the scale loads run one set
    ahead of the operands in their own three-slot ring.  2-3 tiles per CTA
    and K of 2, 3 or 5 blocks make the look-ahead cross tile boundaries, with
    1, 2 or the default number of stages."""
    flags = OFF | fp8g.SINGLE_SM_TILES | (fp8g.STAGES(stages) if stages else 0)
    check_dense_bs(4096, 2048, K, 128, flags, seed=560 + K + stages)


@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("issuers", [0, fp8g.TWO_MMA_ISSUERS, fp8g.ONE_MMA_ISSUER])
def test_dense_pair_many_tiles_and_k_blocks(issuers, gran):
    """Several whole waves of SM-pair tiles and a K of 33 blocks (the scale
    ring wraps many times, 128-element groups span K-block quadruples)."""
    check_dense_bs(1024, 1792, 4224, gran, OFF | fp8g.PAIR_TILES | issuers, seed=530 + gran)


@pytest.mark.parametrize("tn", [2, 3])
def test_pair_narrow_tiles_two_issuers(tn):
    """SM-pair tiles of 64 / 96 columns: two issuers with two buffers each."""
    check_dense_bs(640, 704, 1536, 128, OFF | fp8g.PAIR_TILES | fp8g.TILE_N(tn), seed=533 + tn)


@pytest.mark.parametrize("fa,fb", [(E5, E4), (E4, E5), (E5, E5)])
def test_dense_mixed_formats(fa, fb):
    check_dense_bs(200, 272, 640, 32, OFF, seed=530 + 2 * fa + fb, fa=fa, fb=fb)


@pytest.mark.parametrize("fa,fb", [(E5, E4), (E4, E5), (E5, E5)])
def test_single_sm_scale_ring_mixed_formats(fa, fb):
    # 128-element groups on single-SM tiles: the scale ring with E5M2 operands
    check_dense_bs(384, 672, 1664, 128, OFF | fp8g.SINGLE_SM_TILES, seed=570 + 2 * fa + fb, fa=fa, fb=fb)


@pytest.mark.parametrize("kernel", ["pair", "single_sm"])
def test_dense_one_stage_pipeline(kernel):
    # one stage: a single MMA issuer (two need an even stage count)
    check_dense_bs(256, 384, 1024, 128, DENSE_KERNELS[kernel] | fp8g.DEBUG_ONE_STAGE, seed=535)


@pytest.mark.parametrize("flags", [OFF | fp8g.SINGLE_SM_TILES, ON])
@pytest.mark.parametrize("stages", [2, 3, 5])
def test_short_pipelines(stages, flags):
    # stage caps: two issuers run on the largest even count below the cap
    M = 40 if flags == ON else 256
    check_dense_bs(M, 384, 1536, 128, flags | fp8g.STAGES(stages), seed=536 + stages)


def test_exact_data_is_bit_exact():
    """Small-integer operands and power-of-two scales: every partial sum is
    exact in FP32, so the result must equal the oracle bit for bit."""
    M, N, K = 256, 320, 512
    rng = np.random.default_rng(540)
    vals = np.array([-2.0, -1.0, 0.0, 1.0, 2.0])
    A = synth.encode_fp8_array(vals[rng.integers(0, 5, (M, K))], E4)
    B = synth.encode_fp8_array(vals[rng.integers(0, 5, (N, K))], E4)
    for gran in (128, 32):
        ks = K // gran
        sfa = ue8m0((ks, M), 541 + gran, 124, 130)
        sfb = ue8m0((ks, N), 542 + gran, 124, 130)
        for flags in (OFF | fp8g.PAIR_TILES, OFF | fp8g.SINGLE_SM_TILES, ON):
            D = fp8g.fp8_gemm_nt_blockscaled(dev(A), dev(B), dev(sfa), dev(sfb), sf_group_k=gran,
                                             a_dtype=E4, b_dtype=E4, flags=flags)
            torch.cuda.synchronize()
            assert_status_ok()
            ref, _ = oracle.gemm_blockscaled(A, B, sfa, sfb, gran)
            assert np.array_equal(bits(D), ref), (gran, flags)


def test_scales_reach_the_right_k_group():
    """One K group scaled 2^20 above the rest: the result is (to BF16
    precision) that group's product alone, for every group position."""
    M, N, K = 128, 256, 640
    A = synth.normal_fp8((M, K), 545, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 546, 0.0, 1.0, E4)
    for gran in (128, 32):
        ks = K // gran
        for j in (0, 1, ks - 1):
            sfa = np.full((ks, M), 107, np.uint8)
            sfa[j] = 127
            sfb = np.full((ks, N), 127, np.uint8)
            for flags in (OFF | fp8g.PAIR_TILES, OFF | fp8g.SINGLE_SM_TILES, ON):
                D = fp8g.fp8_gemm_nt_blockscaled(dev(A), dev(B), dev(sfa), dev(sfb), sf_group_k=gran,
                                                 a_dtype=E4, b_dtype=E4, flags=flags)
                torch.cuda.synchronize()
                assert_status_ok()
                ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, want_accbound=True)
                ok, rep = oracle.check_bf16(bits(D), ref, absdot, acc_bound=accb)
                assert ok, (gran, j, flags, rep)


# ---- SwapAB (weights on M, tokens on the runtime N) -----------------------------------

@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("flags", [ON, ON | fp8g.WHOLE_TILES, ON | fp8g.ONE_MMA_ISSUER])
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (40, 640, 1536), (100, 384, 4112), (224, 512, 1024)])
def test_swap(M, N, K, flags, gran):
    # Token chunks of 16, 48 and 112 take two MMA issuers (alternate K blocks,
    # two accumulators); 224 takes one.  (1, 256, 512): eight CTAs of one K
    # block each, so a segment's second accumulator is often empty.
    check_dense_bs(M, N, K, gran, flags, seed=550 + M + N + gran)


@pytest.mark.parametrize("M", [1, 16, 33, 64, 130])
def test_auto_small_m(M):
    check_dense_bs(M, 2048, 1024, 128, AUTO, seed=560 + M)


# ---- masked grouped -------------------------------------------------------------------

def grouped_bs_case(G, M_max, N, K, mm, gran, flags, hint, seed, fa=E4, fb=E4):
    A = synth.normal_fp8((G, M_max, K), seed, 0.0, 0.5, fa)
    B = synth.normal_fp8((G, N, K), seed + 1, 0.0, 0.5, fb)
    mm = np.asarray(mm, np.int32)
    ks = -(-K // gran)
    sfa = ue8m0((G, ks, ld16(M_max)), seed + 2)
    sfb = ue8m0((G, ks, ld16(N)), seed + 3)
    for g in range(G):                      # padding tokens: NaN data and NaN scales
        A[g, mm[g]:] = 0x7F
        sfa[g, :, mm[g]:] = 255
    D0 = synth.u16_pattern((G, M_max, N), seed + 4)
    D0[..., ::89] = 0x7FC1
    Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked_blockscaled(dev(A), dev(B), dev(mm), dev(sfa), dev(sfb), D=Dt,
                                             max_m_hint=hint, sf_group_k=gran, a_dtype=fa, b_dtype=fb,
                                             flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    got = bits(Dt)
    ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, masked_m=mm, D_init=D0, fa=fa, fb=fb,
                                                want_accbound=True)
    for g in range(G):
        m = mm[g]
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m], acc_bound=accb[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g


@pytest.mark.parametrize("gran", [128, 32])
@pytest.mark.parametrize("flags,hint", [(ON, 32), (ON | fp8g.WHOLE_TILES, 64), (ON | fp8g.ONE_MMA_ISSUER, 32),
                                        (ON | fp8g.TOKEN_BOX(16), 32), (OFF, 0), (AUTO, 0)])
def test_grouped(flags, hint, gran):
    mm = [0, 1, 9, 16, 17, 32, 5, 64]
    grouped_bs_case(len(mm), 64, 384, 640, mm, gran, flags, hint, seed=600 + gran)


def test_grouped_mixed_formats():
    grouped_bs_case(3, 48, 256, 512, [48, 7, 0], 128, ON, 48, seed=610, fa=E5, fb=E4)


def test_grouped_moe_decode_shape():
    G, M_max, N, K = 8, 128, 4096, 7168
    mm = [3, 64, 0, 17, 40, 1, 8, 128]
    grouped_bs_case(G, M_max, N, K, mm, 128, AUTO, 0, seed=620)


# ---- host-side argument checks (no kernel runs) -------------------------------------

def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def test_argument_errors():
    lib = _lib.load()
    A = torch.zeros((64, 256), dtype=torch.uint8, device="cuda")
    B = torch.zeros((48, 256), dtype=torch.uint8, device="cuda")
    D = torch.zeros((64, 48), dtype=torch.bfloat16, device="cuda")
    s = torch.full((4096,), 127, dtype=torch.uint8, device="cuda")

    def call(sa, lda, sb, ldb, gran):
        return lib.fp8_gemm_nt_blockscaled(_ptr(A), _ptr(B), _ptr(D), 64, 48, 256, 0, 0, sa, lda, sb, ldb,
                                           gran, 0, None)
    assert call(_ptr(s), 64, _ptr(s), 48, 128) == fp8g.OK
    assert call(_ptr(s), 64, _ptr(s), 48, 32) == fp8g.OK
    assert call(None, 64, _ptr(s), 48, 128) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 64, None, 48, 128) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 64, _ptr(s), 48, 64) == fp8g.ERR_INVALID_ARG
    assert call(_ptr(s), 48, _ptr(s), 48, 128) == fp8g.ERR_INVALID_ARG      # lda < M
    assert call(_ptr(s), 64, _ptr(s), 32, 128) == fp8g.ERR_INVALID_ARG      # ldb < N
    assert call(_ptr(s), 72, _ptr(s), 48, 128) == fp8g.ERR_MISALIGNED       # lda % 16
    off = ctypes.c_void_p(s.data_ptr() + 8)
    assert call(off, 64, _ptr(s), 48, 128) == fp8g.ERR_MISALIGNED
    torch.cuda.synchronize()
    assert_status_ok()
    with pytest.raises(ValueError):
        fp8g.fp8_gemm_nt_blockscaled(A, B, s[:128].view(2, 64), s[:96].view(2, 48), a_dtype=E4, b_dtype=E4,
                                     sf_group_k=32)
