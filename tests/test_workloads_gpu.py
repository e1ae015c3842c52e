"""Parity at the benchmark workloads' full sizes, with the bench's own input
recipes and launch flags: every element of every workload (4096^3, the
eight M=8192 projection runs, the masked MoE-decode workload, every small-M
case and the block-scaled forms) against the oracle, the larger ones one
block of output rows at a time."""
import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import bench
import fp8_tensor_core_gb300 as fp8g
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()
    torch.cuda.set_device(0)
    fp8g.fp8g_get_device_status()
    yield


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_dense_workload(w):
    inp = bench.host_inputs(w)
    A = torch.from_numpy(inp["A"]).cuda()
    B = torch.from_numpy(inp["B"]).cuda()
    D = fp8g.fp8_gemm_nt(A, B, a_dtype=w.fa, b_dtype=w.fb, flags=w.flags)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    return inp, bits(D)


def test_dense4096_every_element():
    w = bench.make_workload("dense4096")
    inp, got = run_dense_workload(w)
    ref, absdot = oracle.gemm_nt(inp["A"], inp["B"], w.fa, w.fb)
    ok, rep = oracle.check_bf16(got, ref, absdot)
    assert ok, rep


PROJ = ["proj:7168:2048", "proj:4096:7168", "proj:18432:7168", "proj:7168:18432"]
ROW_BLOCK = 1024     # oracle rows per call: bounds the host memory of the reference and its sums


@pytest.mark.parametrize("name", PROJ + [p + ":e5m2" for p in PROJ])
def test_projection_every_element(name):
    """The M=8192 projections, B in E4M3 and in E5M2: every element of D
    against the oracle (all host cores), one block of rows at a time."""
    w = bench.make_workload(name)
    inp, got = run_dense_workload(w)
    for r0 in range(0, w.M, ROW_BLOCK):
        r1 = min(w.M, r0 + ROW_BLOCK)
        ref, absdot = oracle.gemm_nt(inp["A"][r0:r1], inp["B"], w.fa, w.fb, nthreads=0)
        ok, rep = oracle.check_bf16(got[r0:r1], ref, absdot)
        assert ok, (r0, rep)


def test_masked_moe_decode_every_valid_row_and_untouched_padding():
    w = bench.make_workload("masked")
    inp = bench.host_inputs(w)
    mm = inp["masked_m"]
    D0 = np.full((w.G, w.M_max, w.N), 0x7FC3, np.uint16)      # NaN canaries everywhere
    Dt = torch.from_numpy(D0.view(np.int16)).cuda().view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked(torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["B"]).cuda(),
                                 torch.from_numpy(mm).cuda(), D=Dt, max_m_hint=w.hint,
                                 a_dtype=w.fa, b_dtype=w.fb, flags=w.flags)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    got = bits(Dt)
    ref, absdot = oracle.gemm_grouped_masked(inp["A"], inp["B"], mm, D0, w.fa, w.fb)
    for g in range(w.G):
        m = int(mm[g])
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g


SMALLM = ["smallm:%d:%s:%s" % (m, nk, mode) for nk in ("24576:1536", "7168:16384")
          for m in (1, 8, 16, 32, 64) for mode in ("swap", "noswap")]
# token counts off the 16-row grid (TMA boxes of exactly the rows) and the
# library's own choice
SMALLM += ["smallm:17:7168:16384:swap", "smallm:33:24576:1536:noswap", "smallm:100:24576:1536:noswap",
           "smallm:5:7168:16384", "smallm:64:24576:1536"]


@pytest.mark.parametrize("name", SMALLM)
def test_small_m_every_element(name):
    w = bench.make_workload(name)
    inp, got = run_dense_workload(w)
    ref, absdot = oracle.gemm_nt(inp["A"], inp["B"], w.fa, w.fb)
    ok, rep = oracle.check_bf16(got, ref, absdot)
    assert ok, rep


BLOCKSCALED = ["dense4096:bs", "masked:bs", "masked:bs32", "smallm:16:7168:16384:auto:bs",
               "smallm:64:24576:1536:auto:bs32", "proj:7168:2048:bs", "proj:7168:18432:bs"]


@pytest.mark.parametrize("name", BLOCKSCALED)
def test_blockscaled_workload(name):
    """Block-scaled workloads with the bench's recipes and flags: every
    element (the M=8192 projections one block of rows at a time), padding
    rows of the masked output untouched."""
    w = bench.make_workload(name)
    inp = bench.host_inputs(w)
    sfa, sfb = torch.from_numpy(inp["sf_a"]).cuda(), torch.from_numpy(inp["sf_b"]).cuda()
    A, B = torch.from_numpy(inp["A"]).cuda(), torch.from_numpy(inp["B"]).cuda()
    if w.kind == "dense":
        D = fp8g.fp8_gemm_nt_blockscaled(A, B, sfa, sfb, sf_group_k=w.gran, a_dtype=w.fa, b_dtype=w.fb,
                                         flags=w.flags)
        torch.cuda.synchronize()
        st = fp8g.fp8g_get_device_status()
        assert st[0] == fp8g.OK, st
        got = bits(D)
        for r0 in range(0, w.M, ROW_BLOCK):
            r1 = min(w.M, r0 + ROW_BLOCK)
            ref, absdot, accb = oracle.gemm_blockscaled(inp["A"][r0:r1], inp["B"],
                                                        np.ascontiguousarray(inp["sf_a"][0][:, r0:r1]),
                                                        inp["sf_b"][0], w.gran, fa=w.fa, fb=w.fb, want_accbound=True)
            ok, rep = oracle.check_bf16(got[r0:r1], ref, absdot, acc_bound=accb)
            assert ok, (r0, rep)
        return
    mm = inp["masked_m"]
    D0 = np.full((w.G, w.M_max, w.N), 0x7FC3, np.uint16)
    Dt = torch.from_numpy(D0.view(np.int16)).cuda().view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked_blockscaled(A, B, torch.from_numpy(mm).cuda(), sfa, sfb, D=Dt,
                                             max_m_hint=w.hint, sf_group_k=w.gran, a_dtype=w.fa, b_dtype=w.fb,
                                             flags=w.flags)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    got = bits(Dt)
    ref, absdot, accb = oracle.gemm_blockscaled(inp["A"], inp["B"], inp["sf_a"], inp["sf_b"], w.gran, masked_m=mm,
                                                D_init=D0, fa=w.fa, fb=w.fb, want_accbound=True)
    for g in range(w.G):
        m = int(mm[g])
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m], acc_bound=accb[g, :m])
        assert ok, (g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "padding rows of group %d written" % g
