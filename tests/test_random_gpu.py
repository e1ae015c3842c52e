"""Seeded random problems across every entry point, checked element by
element against the oracle.

The fixed-shape tests pin each kernel, flag and edge case on purpose; these
draw the shapes, formats, token counts, group layouts and forcing flags at
random (one fixed seed, so a failure reproduces), to reach combinations no
one wrote down: ragged M, N and K together, a token count just past a tile,
empty and full groups next to each other, a forced kernel on a shape it
would not have picked.  Sizes are drawn log-uniformly and capped so that the
oracle finishes the lot in seconds.

Acceptance as everywhere: |gpu - oracle| <= ulp_bf16(oracle) + 1e-6 *
sum|a b| per element ("DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核
优化实践" §1.3, FP32 accumulation, BF16 out), plus, for block scales, the
FP32 accumulation-order bound of the oracle's acc_bound; rows outside the
valid tokens of a group keep their bytes."""
import math

import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
import oracle
import synth

E4, E5 = synth.E4M3, synth.E5M2
OFF, ON, AUTO = fp8g.SWAP_OFF, fp8g.SWAP_ON, fp8g.SWAP_AUTO
SEED = 20261202
MAC_CAP = 1.2e9           # multiply-adds per problem
LARGE_MAC_CAP = 12e9      # ... of the large dense ones

DENSE_FLAGS = [AUTO, AUTO, ON, OFF, OFF | fp8g.SINGLE_SM_TILES, OFF | fp8g.STREAM_K, OFF | fp8g.SPLIT_TAIL,
               OFF | fp8g.WHOLE_TILES, ON | fp8g.WHOLE_TILES, ON | fp8g.SHARE_SM, ON | fp8g.NO_SHARE_SM,
               OFF | fp8g.TILE_N(128), OFF | fp8g.TILE_N(160), OFF | fp8g.TILE_N(224), OFF | fp8g.STAGES(2),
               OFF | fp8g.STAGES(3), AUTO | fp8g.DEBUG_ONE_STAGE]
LARGE_FLAGS = [AUTO, AUTO, OFF | fp8g.SPLIT_TAIL, OFF | fp8g.STREAM_K, OFF | fp8g.TILE_N(128) | fp8g.SPLIT_TAIL,
               OFF | fp8g.TILE_N(128), OFF | fp8g.TILE_N(224), OFF | fp8g.WHOLE_TILES, OFF | fp8g.SINGLE_SM_TILES]
GROUPED_FLAGS = [AUTO, AUTO, ON, OFF, OFF | fp8g.PAIR_TILES, ON | fp8g.WHOLE_TILES, OFF | fp8g.STAGES(3)]
CONTIG_FLAGS = [AUTO, ON, OFF]
BS_FLAGS = [AUTO, AUTO, ON, OFF, OFF | fp8g.SINGLE_SM_TILES, OFF | fp8g.PAIR_TILES, OFF | fp8g.ONE_MMA_ISSUER,
            ON | fp8g.ONE_MMA_ISSUER, OFF | fp8g.TWO_MMA_ISSUERS]


def _log_int(rng, lo, hi):
    return int(math.exp(rng.uniform(math.log(lo), math.log(hi + 1))))


def _nk(rng, n_hi=2304, k_hi=6400):
    """N and K, log-uniform; every other draw from the upper eighth of the
    log range up (so that half the problems span many tiles and K blocks)."""
    big = rng.random() < 0.5
    n_lo, k_lo = (n_hi // 64, k_hi // 128) if big else (1, 1)
    return 8 * max(1, _log_int(rng, n_lo, n_hi // 8)), 16 * max(1, _log_int(rng, k_lo, k_hi // 16))


def _counts(rng, G, M_max):
    """Valid rows per group: a mix of empty, full and anything between."""
    mm = rng.integers(0, M_max + 1, G)
    pick = rng.random(G)
    mm[pick < 0.15] = 0
    mm[pick > 0.85] = M_max
    return mm.astype(np.int32)


def _draw(rng, kind):
    """One problem of `kind`, or None when it is over the size caps."""
    fa, fb = int(rng.integers(2)), int(rng.integers(2))
    if kind == "dense":
        # half of them past one 128-row tile (SM pairs, split tails)
        M = _log_int(rng, 1, 1100) if rng.random() < 0.5 else int(rng.integers(129, 1101))
        N, K = _nk(rng)
        if M * N * K > MAC_CAP:
            return None
        return dict(kind=kind, M=M, N=N, K=K, fa=fa, fb=fb, flags=int(rng.choice(DENSE_FLAGS)))
    if kind == "dense_large":
        # many 256-row tiles: whole waves of SM pairs and a split or stream-K tail
        M, N, K = int(rng.integers(1536, 3073)), 8 * int(rng.integers(160, 401)), 16 * int(rng.integers(128, 257))
        if M * N * K > LARGE_MAC_CAP:
            return None
        return dict(kind="dense", M=M, N=N, K=K, fa=fa, fb=fb, flags=int(rng.choice(LARGE_FLAGS)))
    if kind in ("masked", "bs_masked", "scaled_masked"):
        G = int(rng.integers(1, 13))
        M_max = _log_int(rng, 1, 224 if kind == "bs_masked" else 320)
        N, K = _nk(rng, 2048, 4096)
        mm = _counts(rng, G, M_max)
        if int(mm.sum()) * N * K > MAC_CAP or G * M_max * N > 4_000_000:
            return None
        c = dict(kind=kind, G=G, M_max=M_max, N=N, K=K, masked_m=mm, fa=fa, fb=fb,
                 hint=int(rng.choice([0, M_max, int(rng.integers(1, M_max + 1))])))
        if kind == "masked":
            c["flags"] = int(rng.choice(GROUPED_FLAGS))
        elif kind == "bs_masked":
            c.update(gran=int(rng.choice([32, 128])), flags=int(rng.choice([AUTO, ON, OFF])))
        else:
            c.update(per_row=bool(rng.integers(2)), per_col=bool(rng.integers(2)),
                     flags=int(rng.choice([AUTO, ON, OFF, OFF | fp8g.PAIR_TILES])))
        return c
    if kind == "contig":
        G = int(rng.integers(1, 9))
        sizes = _counts(rng, G, _log_int(rng, 1, 300))
        tail = int(rng.integers(0, 40))
        N, K = _nk(rng, 2048, 4096)
        M_total = int(sizes.sum()) + tail
        if M_total < 1 or int(sizes.sum()) * N * K > MAC_CAP:
            return None
        lead = int(rng.integers(0, tail + 1))
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32) + lead
        return dict(kind=kind, G=G, M_total=M_total, N=N, K=K, offsets=off,
                    hint=int(rng.choice([0, int(sizes.max())])) if sizes.max() > 0 else 0,
                    fa=fa, fb=fb, flags=int(rng.choice(CONTIG_FLAGS)))
    M = _log_int(rng, 1, 900) if rng.random() < 0.5 else int(rng.integers(129, 901))
    N, K = _nk(rng, 2048, 4096)
    if M * N * K > MAC_CAP:
        return None
    if kind == "bs":
        return dict(kind=kind, M=M, N=N, K=K, gran=int(rng.choice([32, 128])), fa=fa, fb=fb,
                    flags=int(rng.choice(BS_FLAGS)))
    return dict(kind="epilogue", M=M, N=N, K=K, fa=fa, fb=fb, flags=int(rng.choice(DENSE_FLAGS[:11])),
                per_row=bool(rng.integers(2)), per_col=bool(rng.integers(2)),
                beta=float(rng.choice([0.0, 1.0, -0.5])), bias=bool(rng.integers(2)), relu=bool(rng.integers(2)),
                round_mode=int(rng.integers(4)), alpha=float(rng.choice([1.0, 0.25, -2.0])))


COUNTS = [("dense", 64), ("dense_large", 16), ("masked", 32), ("contig", 16), ("bs", 32), ("bs_masked", 16), ("scaled_masked", 12),
          ("epilogue", 24)]


def make_cases(seed=SEED):
    rng = np.random.default_rng(seed)
    cases = []
    for kind, n in COUNTS:
        got = 0
        while got < n:
            c = _draw(rng, kind)
            if c is not None:
                cases.append(c)
                got += 1
    return cases


CASES = make_cases()


def _case_id(i, c):
    shape = "x".join(str(c[k]) for k in ("G", "M", "M_max", "M_total", "N", "K") if k in c)
    return "%03d-%s-%s-f%x" % (i, c["kind"], shape, c["flags"])


def _plan(c, sms=0, smem=0):
    sf = c.get("gran", 0)
    if c["kind"] in ("dense", "bs", "epilogue"):
        return fp8g.fp8g_describe_plan(fp8g.LAYOUT_DENSE, 1, c["M"], c["N"], c["K"], 0, sf, c["flags"], sms, smem)
    if c["kind"] == "contig":
        return fp8g.fp8g_describe_plan(fp8g.LAYOUT_CONTIGUOUS, c["G"], c["M_total"], c["N"], c["K"], c["hint"], 0,
                                       c["flags"], sms, smem)
    return fp8g.fp8g_describe_plan(fp8g.LAYOUT_MASKED, c["G"], c["M_max"], c["N"], c["K"], c["hint"], sf,
                                   c["flags"], sms, smem)


def test_random_cases_are_accepted_and_varied():
    """Host side: the library plans every drawn case for a 152-SM GB300
    (no argument is rejected), and the draw reaches all three kernels."""
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()          # host planning lives in the library (no GPU needed)
    kernels = set()
    for c in CASES:
        kernels.add(_plan(c, 152, 232448)["kernel"])
    assert kernels == {fp8g.KERNEL_TOKEN_TILES, fp8g.KERNEL_SM_PAIRS, fp8g.KERNEL_SWAP_AB}
    assert sum(c["M" if "M" in c else "G"] * c["N"] * c["K"] for c in CASES if c["kind"] == "dense") > 0


@pytest.fixture(scope="module")
def gpu():
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


def _operands(c, i, shape_a, shape_b):
    A = synth.normal_fp8(shape_a, 7000 + 2 * i, 0.0, 1.0, c["fa"])
    B = synth.normal_fp8(shape_b, 7001 + 2 * i, 0.0, 1.0, c["fb"])
    return A, B


def _scales(rng, shape, ld):
    sf = np.zeros(shape[:-1] + (ld,), np.uint8)
    sf[..., :shape[-1]] = rng.integers(120, 135, shape)
    return sf


def _status_ok():
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(len(CASES)), ids=[_case_id(i, c) for i, c in enumerate(CASES)])
def test_random_case(gpu, i):
    c = CASES[i]
    fa, fb, flags = c["fa"], c["fb"], c["flags"]
    rng = np.random.default_rng(SEED + 1000 + i)
    kind = c["kind"]
    if kind == "dense":
        A, B = _operands(c, i, (c["M"], c["K"]), (c["N"], c["K"]))
        D = fp8g.fp8_gemm_nt(dev(A), dev(B), a_dtype=fa, b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot = oracle.gemm_nt(A, B, fa, fb)
        ok, rep = oracle.check_bf16(bits(D), ref, absdot)
        assert ok, rep
    elif kind == "masked":
        G, M_max, N, K = c["G"], c["M_max"], c["N"], c["K"]
        A, B = _operands(c, i, (G, M_max, K), (G, N, K))
        D0 = synth.u16_pattern((G, M_max, N), SEED + i)
        Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
        fp8g.fp8_gemm_grouped_masked(dev(A), dev(B), dev(c["masked_m"]), D=Dt, max_m_hint=c["hint"], a_dtype=fa,
                                     b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot = oracle.gemm_grouped_masked(A, B, c["masked_m"], D0, fa, fb)
        got = bits(Dt)
        for g, m in enumerate(c["masked_m"]):
            ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
            assert ok, (g, rep)
            assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g
    elif kind == "contig":
        G, M_total, N, K = c["G"], c["M_total"], c["N"], c["K"]
        A, B = _operands(c, i, (M_total, K), (G, N, K))
        D0 = synth.u16_pattern((M_total, N), SEED + i)
        Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
        fp8g.fp8_gemm_grouped_contiguous(dev(A), dev(B), dev(c["offsets"]), D=Dt, max_m_hint=c["hint"], a_dtype=fa,
                                         b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot = oracle.gemm_grouped_contiguous(A, B, c["offsets"], D0, fa, fb)
        got = bits(Dt)
        off = c["offsets"]
        ok, rep = oracle.check_bf16(got[off[0]:off[-1]], ref[off[0]:off[-1]], absdot[off[0]:off[-1]])
        assert ok, rep
        assert np.array_equal(got[:off[0]], D0[:off[0]]) and np.array_equal(got[off[-1]:], D0[off[-1]:]), \
            "rows outside every group written"
    elif kind == "bs":
        M, N, K, gran = c["M"], c["N"], c["K"], c["gran"]
        A, B = _operands(c, i, (M, K), (N, K))
        ks = -(-K // gran)
        lda, ldb = 16 * (-(-M // 16)) + 16 * int(rng.integers(0, 2)), 16 * (-(-N // 16))
        sfa, sfb = _scales(rng, (ks, M), lda), _scales(rng, (ks, N), ldb)
        D = fp8g.fp8_gemm_nt_blockscaled(dev(A), dev(B), dev(sfa), dev(sfb), sf_group_k=gran, a_dtype=fa,
                                         b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, fa=fa, fb=fb, want_accbound=True)
        ok, rep = oracle.check_bf16(bits(D), ref, absdot, acc_bound=accb)
        assert ok, rep
    elif kind == "bs_masked":
        G, M_max, N, K, gran = c["G"], c["M_max"], c["N"], c["K"], c["gran"]
        A, B = _operands(c, i, (G, M_max, K), (G, N, K))
        ks = -(-K // gran)
        sfa = _scales(rng, (G, ks, M_max), 16 * (-(-M_max // 16)))
        sfb = _scales(rng, (G, ks, N), 16 * (-(-N // 16)))
        D0 = synth.u16_pattern((G, M_max, N), SEED + i)
        Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
        fp8g.fp8_gemm_grouped_masked_blockscaled(dev(A), dev(B), dev(c["masked_m"]), dev(sfa), dev(sfb), D=Dt,
                                                 max_m_hint=c["hint"], sf_group_k=gran, a_dtype=fa, b_dtype=fb,
                                                 flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, masked_m=c["masked_m"], D_init=D0,
                                                    fa=fa, fb=fb, want_accbound=True)
        got = bits(Dt)
        for g, m in enumerate(c["masked_m"]):
            ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m], acc_bound=accb[g, :m])
            assert ok, (g, rep)
            assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g
    elif kind == "scaled_masked":
        G, M_max, N, K = c["G"], c["M_max"], c["N"], c["K"]
        A, B = _operands(c, i, (G, M_max, K), (G, N, K))
        sa = np.exp2(rng.uniform(-3, 3, G * M_max if c["per_row"] else G)).astype(np.float32)
        sb = np.exp2(rng.uniform(-3, 3, G * N if c["per_col"] else G)).astype(np.float32)
        D0 = synth.u16_pattern((G, M_max, N), SEED + i)
        Dt = dev(D0.view(np.int16)).view(torch.bfloat16)
        fp8g.fp8_gemm_grouped_masked_scaled(dev(A), dev(B), dev(c["masked_m"]), dev(sa), dev(sb), D=Dt,
                                            max_m_hint=c["hint"], a_dtype=fa, b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        ref, absdot = oracle.gemm_grouped_masked_scaled(A, B, c["masked_m"], sa, sb, D0, fa, fb)
        got = bits(Dt)
        for g, m in enumerate(c["masked_m"]):
            ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
            assert ok, (g, rep)
            assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g
    else:
        M, N, K = c["M"], c["N"], c["K"]
        A, B = _operands(c, i, (M, K), (N, K))
        sa = np.exp2(rng.uniform(-3, 3, M if c["per_row"] else 1)).astype(np.float32)
        sb = np.exp2(rng.uniform(-3, 3, N if c["per_col"] else 1)).astype(np.float32)
        Ct = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to(torch.bfloat16).cuda()
        Cb = Ct.view(torch.int16).cpu().numpy().view(np.uint16)
        bias = rng.standard_normal(N).astype(np.float32) if c["bias"] else None
        epi = {"alpha": c["alpha"], "beta": c["beta"], "relu": c["relu"], "round_mode": c["round_mode"]}
        if c["beta"] != 0.0:
            epi["C"] = Ct
        if bias is not None:
            epi["bias"] = dev(bias)
        D = fp8g.fp8_gemm_nt_ex(dev(A), dev(B), scale_a=dev(sa), scale_b=dev(sb), epilogue=epi, a_dtype=fa,
                                b_dtype=fb, flags=flags)
        torch.cuda.synchronize()
        _status_ok()
        _, absS, S = oracle.gemm_nt(A, B, fa, fb, want_exact=True)
        f = np.broadcast_to(sa.astype(np.float64)[:, None], (M, 1)) * np.broadcast_to(
            sb.astype(np.float64)[None, :], (1, N))
        ref, absdot = oracle.epilogue(S * f, absS * np.abs(f), c["alpha"], c["beta"],
                                      Cb if c["beta"] != 0.0 else None, bias, c["relu"], c["round_mode"])
        ok, rep = oracle.check_bf16(bits(D), ref, absdot)
        assert ok, rep
