"""GPU parity: the CUDA path through the C ABI against the CPU oracle,
element by element, on seeded inputs (small shapes spanning several tiles
and ragged tails, edge cases, then the workload sizes).

Acceptance per element: |gpu - oracle| <= ulp_bf16(oracle) + 1e-6 * sum|a b|
(exactly representable cases must match bit for bit)."""
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
    fp8g.fp8g_get_device_status()      # clear anything left from before
    yield torch.device("cuda:0")


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def assert_status_ok():
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, "device status %s" % (st,)


def dense_inputs(M, N, K, fa, fb, seed, dist="normal", std=1.0):
    if dist == "uniform":
        A = synth.uniform_fp8((M, K), seed, -2.0, 2.0, fa)
        B = synth.uniform_fp8((N, K), seed + 1, -2.0, 2.0, fb)
    else:
        A = synth.normal_fp8((M, K), seed, 0.0, std, fa)
        B = synth.normal_fp8((N, K), seed + 1, 0.0, std, fb)
    return A, B


def run_dense(A, B, fa, fb, flags):
    D = fp8g.fp8_gemm_nt(dev(A), dev(B), a_dtype=fa, b_dtype=fb, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    return bits(D)


def check_dense(M, N, K, fa=E4, fb=E4, flags=AUTO, seed=1, dist="normal", std=1.0):
    A, B = dense_inputs(M, N, K, fa, fb, seed, dist, std)
    got = run_dense(A, B, fa, fb, flags)
    ref, absdot = oracle.gemm_nt(A, B, fa, fb)
    ok, rep = oracle.check_bf16(got, ref, absdot)
    assert ok, rep
    return rep


# ---- first: one tile, then a few -------------------------------------------

@pytest.mark.parametrize("flags", [OFF, ON])
def test_single_tile(flags):
    check_dense(128, 128, 128, flags=flags, seed=11)


@pytest.mark.parametrize("flags", [OFF, ON])
def test_exact_integer_products_bit_exact(flags):
    """Entries in {-2..2}: every partial sum is an integer of magnitude
    <= 256, exact in FP32 and BF16, so the GPU must match bit for bit."""
    rng = np.random.default_rng(5)
    enc = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    M, N, K = 160, 192, 64
    ia = rng.choice([-2, -1, 0, 1, 2], (M, K))
    ib = rng.choice([-2, -1, 0, 1, 2], (N, K))
    A = np.vectorize(enc.get)(ia).astype(np.uint8)
    B = np.vectorize(enc.get)(ib).astype(np.uint8)
    got = run_dense(A, B, E4, E4, flags)
    ref, _ = oracle.gemm_nt(A, B)
    assert np.array_equal(got, ref)


def test_all_ones_K_up_to_256():
    for K in (16, 48, 128, 144, 256):
        A = np.full((130, K), 0x38, np.uint8)
        B = np.full((136, K), 0x38, np.uint8)
        for flags in (OFF, ON):
            got = run_dense(A, B, E4, E4, flags)
            assert np.all(oracle.bf16_bits_to_f64(got) == K), (K, flags)


def test_identity_gives_transpose():
    K, N = 256, 320
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = 0x38
    B = synth.normal_fp8((N, K), 91, 0.0, 1.0, E4)
    for flags in (OFF, ON):
        got = run_dense(A, B, E4, E4, flags)
        ref, _ = oracle.gemm_nt(A, B)
        assert np.array_equal(got, ref)


# ---- shapes: several tiles, ragged tails, K tails -------------------------------

SHAPES = [
    (256, 256, 256),
    (1, 8, 16),
    (7, 24, 48),
    (64, 1024, 384),
    (129, 136, 144),
    (200, 520, 1280),
    (300, 264, 400),
    (513, 776, 272),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("flags", [OFF, ON, AUTO])
def test_dense_shapes(M, N, K, flags):
    check_dense(M, N, K, flags=flags, seed=M * 31 + N * 7 + K)


@pytest.mark.parametrize("M,N,K", [(6144, 6144, 1280), (6145, 6136, 1296), (6143, 6144, 1040)])
def test_dense_page_edge_shapes(M, N, K):
    """The shape of "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
    §6.1 (M = N = 6144, K = 1280, which failed at random there through a
    write past a tile's K tail) and its neighbours: M one row either side of
    a 256-row tile, N 8 short of a tile, K with a 16-byte tail past ten
    128-byte blocks or three quarters of one.  Every element."""
    check_dense(M, N, K, flags=AUTO, seed=M + N + K)


def test_dense_uniform_256_cube():
    """The 256^3 U[-2,2] E4M3 workload, every element."""
    rep = check_dense(256, 256, 256, dist="uniform", seed=synth.seed_for(0))
    assert rep["bad"] == 0


@pytest.mark.parametrize("fa,fb", [(E4, E5), (E5, E4), (E5, E5)])
@pytest.mark.parametrize("flags", [OFF, ON])
def test_mixed_formats(fa, fb, flags):
    check_dense(192, 384, 512, fa=fa, fb=fb, flags=flags, seed=17 + fa * 2 + fb, std=0.5)


@pytest.mark.parametrize("flags", [OFF, ON])
def test_one_stage_pipeline_matches(flags):
    """The one-stage debug pipeline (load, compute, load ...) computes the
    same result as the deep ring."""
    A, B = dense_inputs(150, 264, 640, E4, E4, 23)
    deep = run_dense(A, B, E4, E4, flags)
    one = run_dense(A, B, E4, E4, flags | fp8g.DEBUG_ONE_STAGE)
    assert np.array_equal(deep, one)


def test_accumulator_keeps_small_terms():
    """One product of 256 and 16383 products of 2^-10: the exact sum
    256 + 16383/1024 needs FP32 accumulation; an accumulator that drops the
    small terms returns 256, outside the tolerance."""
    K = 16384
    A = np.full((128, K), 0x10, np.uint8)       # 2^-5
    B = np.full((128, K), 0x10, np.uint8)
    A[:, 0] = 0x58                               # 16
    B[:, 0] = 0x58
    for flags in (OFF, ON):
        got = run_dense(A, B, E4, E4, flags)
        ref, absdot = oracle.gemm_nt(A, B)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, rep
        assert np.all(oracle.bf16_bits_to_f64(got) == 272.0)


def test_deterministic_repeat():
    A, B = dense_inputs(64, 7168, 4096, E4, E4, 29)      # small M: stream-K path
    Ad, Bd = dev(A), dev(B)
    D1 = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4, flags=ON)
    D2 = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4, flags=ON)
    torch.cuda.synchronize()
    assert_status_ok()
    assert torch.equal(D1.view(torch.int16), D2.view(torch.int16))
    ref, absdot = oracle.gemm_nt(A, B)
    ok, rep = oracle.check_bf16(bits(D1), ref, absdot)
    assert ok, rep


def test_side_stream():
    A, B = dense_inputs(256, 512, 512, E4, E4, 37)
    s = torch.cuda.Stream()
    Ad, Bd = dev(A), dev(B)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        D = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4)
    s.synchronize()
    assert_status_ok()
    ref, absdot = oracle.gemm_nt(A, B)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot)
    assert ok, rep


# ---- masked grouped --------------------------------------------------------------

def grouped_case(G, M_max, N, K, mm, flags, hint, seed, nan_padding=False, fa=E4, fb=E4):
    A = synth.normal_fp8((G, M_max, K), seed, 0.0, 0.5, fa)
    B = synth.normal_fp8((G, N, K), seed + 1, 0.0, 0.5, fb)
    mm = np.asarray(mm, np.int32)
    if nan_padding:
        for g in range(G):
            A[g, mm[g]:] = 0x7F
    D0 = synth.u16_pattern((G, M_max, N), seed + 2)
    D0[..., ::97] = 0x7FC1                      # NaN codes among the canaries
    Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked(dev(A), dev(B), dev(mm), D=Dt, max_m_hint=hint,
                                 a_dtype=fa, b_dtype=fb, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    got = bits(Dt)
    ref, absdot = oracle.gemm_grouped_masked(A, B, mm, D0, fa, fb)
    for g in range(G):
        m = mm[g]
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g


@pytest.mark.parametrize("flags,hint", [(OFF | fp8g.PAIR_TILES, 0), (OFF, 0), (AUTO, 640), (OFF, 256),
                                        (OFF | fp8g.PAIR_TILES, 64)])
def test_grouped_pair_tiles(flags, hint):
    """Masked groups of up to 640 tokens on SM-pair tiles: full, partial,
    empty and one-pair-plus-one-row groups, NaN in the padding rows."""
    grouped_case(4, 640, 512, 1024, [640, 300, 0, 129], flags, hint, seed=191, nan_padding=True)


def test_grouped_pair_tiles_mixed_formats_and_narrow_n():
    grouped_case(3, 512, 136, 640, [512, 257, 1], OFF | fp8g.PAIR_TILES, 0, seed=193, fa=E5, fb=E4)


@pytest.mark.parametrize("flags,hint", [(ON, 32), (ON, 0), (OFF, 0), (AUTO, 32), (AUTO, 0)])
def test_grouped_edge_counts(flags, hint):
    mm = [0, 1, 7, 8, 15, 16, 17, 31, 32, 64]
    grouped_case(len(mm), 64, 256, 512, mm, flags, hint, seed=101)


@pytest.mark.parametrize("flags", [ON, OFF])
def test_grouped_nan_padding_never_reaches_valid_rows(flags):
    grouped_case(4, 48, 384, 640, [3, 0, 48, 20], flags, 0, seed=111, nan_padding=True)


def test_grouped_all_empty_writes_nothing():
    grouped_case(3, 32, 128, 256, [0, 0, 0], ON, 16, seed=121)
    grouped_case(3, 32, 128, 256, [0, 0, 0], OFF, 0, seed=122)


def test_grouped_hint_below_actual_counts_is_still_correct():
    grouped_case(5, 96, 256, 384, [90, 3, 40, 96, 17], ON, 16, seed=131)


def test_grouped_masked_m_out_of_range_is_clamped_and_flagged():
    G, M_max, N, K = 3, 32, 128, 256
    A = synth.normal_fp8((G, M_max, K), 141, 0.0, 0.5, E4)
    B = synth.normal_fp8((G, N, K), 142, 0.0, 0.5, E4)
    mm = np.array([-5, 40, 7], np.int32)
    D0 = synth.u16_pattern((G, M_max, N), 143)
    Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked(dev(A), dev(B), dev(mm), D=Dt, a_dtype=E4, b_dtype=E4, flags=ON)
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.ERR_MASKED_M_RANGE
    clamped = np.array([0, 32, 7], np.int32)
    ref, absdot = oracle.gemm_grouped_masked(A, B, clamped, D0)
    got = bits(Dt)
    ok, rep = oracle.check_bf16(got[1], ref[1], absdot[1])
    assert ok, rep
    assert np.array_equal(got[0], D0[0])
    assert_status_ok()


def test_grouped_mixed_formats():
    grouped_case(3, 40, 256, 384, [40, 9, 25], ON, 40, seed=151, fb=E5)


# ---- stream-K partition edge cases (SwapAB kernel) -------------------------------

@pytest.mark.parametrize("M,N,K", [
    (16, 128, 128 * 200),     # one tile whose 200 K blocks span every CTA
    (5, 1280, 128 * 16),      # 160 K blocks over 152 CTAs: ~15 contributors per tile
    (33, 384, 128 * 3),       # fewer K blocks (9) than SMs: partition shrinks
    (64, 24576, 1536),        # the small-M streaming shape, every element
    (1, 7168, 16384),
])
def test_stream_k_partitions(M, N, K):
    check_dense(M, N, K, flags=ON, seed=7 * M + N + K)


def test_whole_tiles_mode_matches_stream_k():
    A, B = dense_inputs(40, 2048, 2048, E4, E4, 41)
    sk = run_dense(A, B, E4, E4, ON)
    wt = run_dense(A, B, E4, E4, ON | fp8g.WHOLE_TILES)
    ref, absdot = oracle.gemm_nt(A, B)
    for got in (sk, wt):
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, rep


def test_grouped_stream_k_many_groups():
    mm = [0, 3, 0, 128, 1, 77, 0, 16, 128, 5, 31, 0]
    grouped_case(len(mm), 128, 384, 1024, mm, ON, 0, seed=161)
    grouped_case(len(mm), 128, 384, 1024, mm, ON | fp8g.WHOLE_TILES, 0, seed=162)


# ---- SM-pair (cta_group::2) dense kernel --------------------------------------------

@pytest.mark.parametrize("M,N,K", [
    (256, 256, 128),          # one 256 x 256 tile
    (257, 224, 384),          # second 256-row tile has one valid row
    (512, 1000, 640),         # ragged N tile
    (384, 96, 1280),          # N narrower than half a tile
    (1024, 2048, 1024),
])
def test_pair_kernel_shapes(M, N, K):
    check_dense(M, N, K, flags=OFF, seed=3 * M + N + K)


def test_pair_matches_single_sm_tiles_bitwise_on_exact_data():
    """Integer-valued data: both kernels are exact, so bit-identical."""
    rng = np.random.default_rng(8)
    enc = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    M, N, K = 600, 736, 64
    A = np.vectorize(enc.get)(rng.choice([-2, -1, 0, 1, 2], (M, K))).astype(np.uint8)
    B = np.vectorize(enc.get)(rng.choice([-2, -1, 0, 1, 2], (N, K))).astype(np.uint8)
    pair = run_dense(A, B, E4, E4, OFF)
    single = run_dense(A, B, E4, E4, OFF | fp8g.SINGLE_SM_TILES)
    ref, _ = oracle.gemm_nt(A, B)
    assert np.array_equal(pair, ref) and np.array_equal(single, ref)


def test_pair_one_stage_and_tile_overrides():
    A, B = dense_inputs(300, 520, 768, E4, E4, 47)
    ref, absdot = oracle.gemm_nt(A, B)
    for flags in (OFF | fp8g.DEBUG_ONE_STAGE, OFF | fp8g.TILE_N(128), OFF | fp8g.TILE_N(256),
                  OFF | fp8g.TILE_N(160)):
        got = run_dense(A, B, E4, E4, flags)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, (hex(flags), rep)


@pytest.mark.parametrize("M,N,K", [
    (256, 256, 128 * 40),     # one tile, 40 K blocks over 76 pairs: 40 contributors
    (512, 512, 128 * 3),      # 4 tiles x 3 K blocks < 76 pairs: partition shrinks
    (1000, 1032, 2000),       # ragged everywhere (K tail of 80 bytes)
])
def test_pair_stream_k_partitions(M, N, K):
    check_dense(M, N, K, flags=OFF | fp8g.STREAM_K, seed=5 * M + N + K)


def test_pair_whole_tiles_and_stream_k_agree():
    A, B = dense_inputs(768, 1280, 1536, E4, E4, 53)
    ref, absdot = oracle.gemm_nt(A, B)
    for flags in (OFF, OFF | fp8g.STREAM_K, OFF | fp8g.STREAM_K | fp8g.TILE_N(256),
                  OFF | fp8g.TILE_N(224)):
        got = run_dense(A, B, E4, E4, flags)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, (hex(flags), rep)


@pytest.mark.parametrize("M,N,K", [(16, 2048, 4096), (128, 1024, 1536), (1, 7168, 2048)])
def test_share_sm_mode_dense(M, N, K):
    check_dense(M, N, K, flags=ON | fp8g.SHARE_SM, seed=11 * M + N + K)


@pytest.mark.parametrize("M", [1, 9, 16])
def test_dense_up_to_16_tokens_with_and_without_sharing(M):
    # the default shares the SM for up to 16 tokens; NO_SHARE_SM keeps the whole SM
    check_dense(M, 3072, 5120, flags=ON, seed=13 * M)
    check_dense(M, 3072, 5120, flags=ON | fp8g.NO_SHARE_SM, seed=13 * M)


@pytest.mark.parametrize("box", [16, 32, 64, 128])
def test_swap_token_box_sizes(box):
    # one 128-token chunk loaded as 128 / box TMA copies per K block
    check_dense(128, 1536, 1024, flags=ON | fp8g.NO_SHARE_SM | fp8g.TOKEN_BOX(box), seed=700 + box)
    check_dense(101, 1536, 1024, flags=ON | fp8g.NO_SHARE_SM | fp8g.TOKEN_BOX(box), seed=800 + box)


@pytest.mark.parametrize("M,flags", [(5, OFF), (5, ON), (21, ON), (100, OFF)])
def test_few_tokens_after_nan_padded_launches(M, flags):
    # Dense problems of few tokens load only their rows; the MMA's remaining
    # rows read whatever earlier launches left in shared memory.  Fill it
    # first with NaN token rows (masked padding over every SM), then check
    # the valid outputs.
    G, M_max, N, K = 32, 128, 512, 1024
    A = np.full((G, M_max, K), 0x7F, np.uint8)
    A[:, 0] = synth.normal_fp8((G, K), 961, 0.0, 0.5, E4)
    B = synth.normal_fp8((G, N, K), 962, 0.0, 0.5, E4)
    mm = np.ones(G, np.int32)
    Dg = torch.empty((G, M_max, N), dtype=torch.bfloat16, device="cuda:0")
    for mode in (ON, OFF):
        fp8g.fp8_gemm_grouped_masked(dev(A), dev(B), dev(mm), D=Dg, max_m_hint=M_max, a_dtype=E4, b_dtype=E4,
                                     flags=mode | fp8g.WHOLE_TILES)
    check_dense(M, 3072, 2048, flags=flags, seed=963 + M)


@pytest.mark.parametrize("M2,flags", [(8, AUTO), (64, AUTO), (32, OFF)])
def test_weights_written_by_the_previous_launch_are_seen(M2, flags):
    # GEMM 1 writes its BF16 output into the bytes GEMM 2 then reads as FP8
    # weights, launched right before it on the same stream.  Dense launches
    # fetch weights into L2 before waiting for the previous launch; the
    # product must still use what GEMM 1 wrote, never the stale contents.
    # GEMM 1 gathers finite E4M3 values (one-hot A rows times B1), so D1 is
    # exact and its bytes are finite E4M3 codes.
    N2, K2 = 2048, 4096
    M1, N1, K1 = N2, K2 // 2, 32
    A1 = np.zeros((M1, K1), np.uint8)
    A1[np.arange(M1), np.arange(M1) % K1] = 0x38            # 1.0
    B1 = synth.normal_fp8((N1, K1), 951, 0.0, 1.0, E4)
    A2 = synth.normal_fp8((M2, K2), 952, 0.0, 1.0, E4)
    D1 = torch.full((M1, N1), 1.5, dtype=torch.bfloat16, device="cuda:0")   # stale bytes 0x3F, 0xC0
    a1, b1, a2 = dev(A1), dev(B1), dev(A2)
    torch.cuda.synchronize()
    fp8g.fp8_gemm_nt(a1, b1, D=D1, a_dtype=E4, b_dtype=E4)
    D2 = fp8g.fp8_gemm_nt(a2, D1.view(torch.uint8), a_dtype=E4, b_dtype=E4, flags=flags)
    torch.cuda.synchronize()
    assert_status_ok()
    B2 = D1.view(torch.uint8).cpu().numpy()
    ref1, _ = oracle.gemm_nt(A1, B1, E4, E4)
    assert np.array_equal(B2.view(np.uint16), ref1), "GEMM 1 output"
    ref, absdot = oracle.gemm_nt(A2, B2, E4, E4)
    ok, rep = oracle.check_bf16(bits(D2), ref, absdot)
    assert ok, rep


def test_share_sm_mode_grouped():
    mm = [0, 5, 32, 17, 1, 64]
    grouped_case(len(mm), 64, 512, 1024, mm, ON | fp8g.SHARE_SM, 32, seed=171)


def test_init_then_capture_stream_k_in_a_graph():
    """After fp8g_init on a stream, a stream-K call on that stream allocates
    nothing, so it can be the first call recorded into a CUDA graph captured
    from it; fp8g_shutdown frees the workspaces and later calls allocate
    them again."""
    fp8g.fp8g_shutdown()
    M, N, K = 24, 1536, 3072
    A = synth.normal_fp8((M, K), 181, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 182, 0.0, 1.0, E4)
    Ad, Bd = dev(A), dev(B)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    fp8g.fp8g_init(0, s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fp8g.fp8_gemm_nt(Ad, Bd, D, a_dtype=E4, b_dtype=E4, flags=ON)
    g.replay()
    torch.cuda.synchronize()
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
    ref, absdot = oracle.gemm_nt(A, B)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot)
    assert ok, rep
    fp8g.fp8g_shutdown()
    D2 = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4, flags=ON)
    torch.cuda.synchronize()
    ok, rep = oracle.check_bf16(bits(D2), ref, absdot)
    assert ok, rep


def test_init_argument_errors():
    assert fp8g._lib.load().fp8g_init(-1, None) == fp8g.ERR_INVALID_ARG
    assert fp8g._lib.load().fp8g_init(1 << 40, None) == fp8g.ERR_INVALID_ARG


def test_release_stream_frees_and_later_calls_allocate_again():
    """fp8g_release_stream synchronises the stream and frees its workspace;
    the next stream-K call on it allocates a fresh one and is still right."""
    M, N, K = 40, 2048, 2048
    A = synth.normal_fp8((M, K), 191, 0.0, 1.0, E4)
    B = synth.normal_fp8((N, K), 192, 0.0, 1.0, E4)
    Ad, Bd = dev(A), dev(B)
    ref, absdot = oracle.gemm_nt(A, B)
    s = torch.cuda.Stream()
    for _ in range(2):
        with torch.cuda.stream(s):
            D = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=E4, b_dtype=E4, flags=ON)
        fp8g.fp8g_release_stream(s)
        ok, rep = oracle.check_bf16(bits(D), ref, absdot)
        assert ok, rep
    fp8g.fp8g_release_stream(s)          # nothing left to free: still OK
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK
