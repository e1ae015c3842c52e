"""Library calls on unordered streams, running at the same time on the GPU.

The SwapAB kernel splits K blocks evenly over the CTAs (stream-K) and sums a
tile's FP32 partial tiles through scratch memory ("DeepGEMM：基于 Hopper Tensor
Core 的 FP8 矩阵乘法内核优化实践" §6.4 warns about accumulation across CTAs).
Each stream has its own scratch, so two streams' launches may overlap.  Here
the masked MoE-decode workload (SwapAB, stream 1) and a 16-token dense
small-M problem (SwapAB stream-K, stream 2) are enqueued many times with no
ordering between the streams, each call into an output buffer of its own;
every valid element of every call is checked against the oracle and the
padding rows of the masked outputs must stay untouched bit for bit."""
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


def check_dense(got, ref, absdot, what):
    ok, rep = oracle.check_bf16(got, ref, absdot)
    assert ok, (what, rep)


def check_masked(got, D0, ref, absdot, mm, what):
    for g in range(mm.size):
        m = int(mm[g])
        ok, rep = oracle.check_bf16(got[g, :m], ref[g, :m], absdot[g, :m])
        assert ok, (what, g, rep)
        assert np.array_equal(got[g, m:], D0[g, m:]), "%s: padding rows of group %d written" % (what, g)


@pytest.mark.parametrize("small", ["smallm:16:7168:16384:swap", "smallm:64:24576:1536:swap"])
def test_stream_k_calls_on_unordered_streams(small):
    wm = bench.make_workload("masked")        # SwapAB (the configured path), stream-K
    ws = bench.make_workload(small)
    assert wm.flags & 3 == fp8g.SWAP_ON and ws.flags & 3 == fp8g.SWAP_ON
    for w, kind in ((wm, fp8g.LAYOUT_MASKED), (ws, fp8g.LAYOUT_DENSE)):
        plan = bench.planned_launch(w)
        assert plan["kernel"] == fp8g.KERNEL_SWAP_AB and plan["stream_k"] == 1, plan

    im, is_ = bench.host_inputs(wm), bench.host_inputs(ws)
    mm = im["masked_m"]
    Am, Bm, mmd = (torch.from_numpy(im[k]).cuda() for k in ("A", "B", "masked_m"))
    As, Bs = torch.from_numpy(is_["A"]).cuda(), torch.from_numpy(is_["B"]).cuda()
    D0 = np.full((wm.G, wm.M_max, wm.N), 0x7FC3, np.uint16)      # NaN canaries
    D0_t = torch.from_numpy(D0.view(np.int16)).cuda()

    n_masked, per_masked = 6, 5          # ~140 us masked launches, 10-30 us small ones
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Dm = [D0_t.clone().view(torch.bfloat16) for _ in range(n_masked)]
    Ds = [torch.full((ws.M, ws.N), float("nan"), dtype=torch.bfloat16, device="cuda")
          for _ in range(n_masked * per_masked)]
    start = torch.cuda.Event()
    torch.cuda.synchronize()
    start.record(torch.cuda.current_stream())
    s1.wait_event(start)
    s2.wait_event(start)
    for r in range(n_masked):
        fp8g.fp8_gemm_grouped_masked(Am, Bm, mmd, D=Dm[r], max_m_hint=wm.hint, a_dtype=wm.fa, b_dtype=wm.fb,
                                     flags=wm.flags, stream=s1)
        for j in range(per_masked):
            fp8g.fp8_gemm_nt(As, Bs, Ds[r * per_masked + j], a_dtype=ws.fa, b_dtype=ws.fb, flags=ws.flags,
                             stream=s2)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st

    ref_m, abs_m = oracle.gemm_grouped_masked(im["A"], im["B"], mm, D0, wm.fa, wm.fb)
    ref_s, abs_s = oracle.gemm_nt(is_["A"], is_["B"], ws.fa, ws.fb)
    for r in range(n_masked):
        check_masked(bits(Dm[r]), D0, ref_m, abs_m, mm, "masked call %d" % r)
    for i, D in enumerate(Ds):
        check_dense(bits(D), ref_s, abs_s, "small-M call %d" % i)


def test_split_pair_tiles_and_swap_on_unordered_streams():
    """The 4096^3 dense GEMM, whose last partial wave is split along K (its
    contributors publish FP32 partial tiles through the stream's scratch),
    on one stream and 16-token SwapAB stream-K calls on another, with no
    ordering between them: every element of every call against the oracle."""
    wd = bench.make_workload("dense4096")
    ws = bench.make_workload("smallm:16:7168:16384:swap")
    plan = bench.planned_launch(wd)
    assert plan["kernel"] == fp8g.KERNEL_SM_PAIRS and plan["stream_k"] == 1, plan
    idn, is_ = bench.host_inputs(wd), bench.host_inputs(ws)
    Ad, Bd = torch.from_numpy(idn["A"]).cuda(), torch.from_numpy(idn["B"]).cuda()
    As, Bs = torch.from_numpy(is_["A"]).cuda(), torch.from_numpy(is_["B"]).cuda()
    n_dense, per_dense = 6, 2
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Dd = [torch.full((wd.M, wd.N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(n_dense)]
    Ds = [torch.full((ws.M, ws.N), float("nan"), dtype=torch.bfloat16, device="cuda")
          for _ in range(n_dense * per_dense)]
    start = torch.cuda.Event()
    torch.cuda.synchronize()
    start.record(torch.cuda.current_stream())
    s1.wait_event(start)
    s2.wait_event(start)
    for r in range(n_dense):
        fp8g.fp8_gemm_nt(Ad, Bd, Dd[r], a_dtype=wd.fa, b_dtype=wd.fb, flags=wd.flags, stream=s1)
        for j in range(per_dense):
            fp8g.fp8_gemm_nt(As, Bs, Ds[r * per_dense + j], a_dtype=ws.fa, b_dtype=ws.fb, flags=ws.flags,
                             stream=s2)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    ref_d, abs_d = oracle.gemm_nt(idn["A"], idn["B"], wd.fa, wd.fb)
    ref_s, abs_s = oracle.gemm_nt(is_["A"], is_["B"], ws.fa, ws.fb)
    first = bits(Dd[0])
    for r in range(n_dense):
        got = bits(Dd[r])
        check_dense(got, ref_d, abs_d, "dense call %d" % r)
        assert np.array_equal(got, first), "dense call %d differs from the first" % r
    for i, D in enumerate(Ds):
        check_dense(bits(D), ref_s, abs_s, "small-M call %d" % i)
