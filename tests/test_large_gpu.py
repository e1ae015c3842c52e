"""64-bit addressing on the GPU: buffers whose byte offsets pass 2^32 (the
invariant behind "MLS 三个访存 Bug 深度剖析", Bug 1: a carry lost in 32-bit
address arithmetic shifts accesses by 4 GiB).  Outputs past the 4 GiB mark
are compared with the oracle.  The big tensors repeat small seeded blocks
(replicated on the device), so the oracle sees exactly the host blocks."""
import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
import oracle
import synth

pytestmark = pytest.mark.gpu

FOUR_GIB = 1 << 32


@pytest.fixture(scope="module", autouse=True)
def device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()
    torch.cuda.set_device(0)
    fp8g.fp8g_get_device_status()
    yield
    torch.cuda.empty_cache()


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("flags", [fp8g.SWAP_OFF, fp8g.SWAP_OFF | fp8g.SINGLE_SM_TILES])
def test_output_offsets_past_4gib(flags):
    M, N, K = 140_000, 16384, 128            # D = 4.59 GB of BF16
    assert M * N * 2 > FOUR_GIB
    block = synth.normal_fp8((1000, K), 701, 0.0, 1.0, synth.E4M3)
    B = synth.normal_fp8((N, K), 702, 0.0, 1.0, synth.E4M3)
    reps = -(-M // 1000)
    A_dev = torch.from_numpy(block).cuda().repeat(reps, 1)[:M].contiguous()
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8g.fp8_gemm_nt(A_dev, torch.from_numpy(B).cuda(), D, a_dtype=0, b_dtype=0, flags=flags)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    rows = np.array([M - 1, M - 2, 131_072, 131_071, 139_999 - 500, 0])
    assert (rows.max() * N * 2) > FOUR_GIB
    got = bits(D[torch.from_numpy(rows).cuda()])
    ref, absdot = oracle.gemm_nt(block[rows % 1000], B)
    ok, rep = oracle.check_bf16(got, ref, absdot)
    assert ok, rep
    del D, A_dev


def test_grouped_weights_past_4gib():
    G, M_max, N, K = 40, 32, 16384, 7168      # B = 4.70 GB
    assert G * N * K > FOUR_GIB
    blocks = synth.normal_fp8((4, N, K), 711, 0.0, 0.5, synth.E4M3)       # 470 MB on the host
    A = synth.normal_fp8((G, M_max, K), 712, 0.0, 0.5, synth.E4M3)
    mm = np.array([(g * 7) % 33 for g in range(G)], np.int32)
    mm[-1], mm[-2] = 32, 17
    blk = torch.from_numpy(blocks).cuda()
    B_dev = torch.empty((G, N, K), dtype=torch.uint8, device="cuda")
    for g in range(G):
        B_dev[g].copy_(blk[g % 4])
    del blk
    D0 = np.full((G, M_max, N), 0x7FC5, np.uint16)
    Dt = torch.from_numpy(D0.view(np.int16)).cuda().view(torch.bfloat16)
    fp8g.fp8_gemm_grouped_masked(torch.from_numpy(A).cuda(), B_dev, torch.from_numpy(mm).cuda(), Dt,
                                 max_m_hint=32, a_dtype=0, b_dtype=0, flags=fp8g.SWAP_ON)
    torch.cuda.synchronize()
    st = fp8g.fp8g_get_device_status()
    assert st[0] == fp8g.OK, st
    got = bits(Dt)
    for g in (G - 1, G - 2, 0):
        m = int(mm[g])
        ref, absdot = oracle.gemm_nt(A[g, :m], blocks[g % 4])
        ok, rep = oracle.check_bf16(got[g, :m], ref, absdot)
        assert ok, (g, rep)
        assert np.all(got[g, m:] == 0x7FC5)
    del B_dev, Dt
