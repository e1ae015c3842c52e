"""Failure detection on the GPU without a fault: every barrier wait in the
kernels is bounded.  FP8G_DEBUG_DROP_FIRST_LOAD makes block 0 skip its first
copy, so a wait that nothing will satisfy runs out; the kernel must record
FP8G_ERR_TIMEOUT in the device status word, drain, free its tensor memory
and return, leaving the context usable for the next, correct call."""
import time

import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import fp8_tensor_core_gb300 as fp8g
import oracle
import synth

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000          # 20 ms per wait in these launches


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


@pytest.mark.parametrize("M,N,K,flags,name", [
    (512, 768, 1024, fp8g.SWAP_OFF, "SM-pair kernel"),
    (128, 512, 1024, fp8g.SWAP_OFF, "single-SM kernel"),
    (32, 2048, 2048, fp8g.SWAP_ON, "SwapAB stream-K kernel"),
])
def test_wait_runs_out_then_gpu_still_correct(M, N, K, flags, name):
    A = synth.normal_fp8((M, K), 601 + M, 0.0, 1.0, synth.E4M3)
    B = synth.normal_fp8((N, K), 602 + N, 0.0, 1.0, synth.E4M3)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    prev = fp8g.fp8g_set_wait_timeout_ns(LIMIT_NS)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=0, b_dtype=0, flags=flags | fp8g.DEBUG_DROP_FIRST_LOAD)
        st = fp8g.fp8g_get_device_status()
        elapsed = time.perf_counter() - t0
    finally:
        fp8g.fp8g_set_wait_timeout_ns(prev)
    assert st[0] == fp8g.ERR_TIMEOUT, (name, st)
    assert st[1] in (0, 1), st                      # block 0 (or its pair peer)
    assert elapsed < 5.0, elapsed                   # bounded: far below a hang
    # The context is still healthy: the same call without the injected drop
    # matches the oracle and records no error.
    D = fp8g.fp8_gemm_nt(Ad, Bd, a_dtype=0, b_dtype=0, flags=flags)
    st2 = fp8g.fp8g_get_device_status()
    assert st2[0] == fp8g.OK, st2
    ref, absdot = oracle.gemm_nt(A, B)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot)
    assert ok, (name, rep)


def test_status_word_is_cleared_by_reading():
    assert fp8g.fp8g_get_device_status()[0] == fp8g.OK


@pytest.mark.parametrize("M,N,K,flags,name", [
    (512, 768, 1024, fp8g.SWAP_OFF | fp8g.PAIR_TILES, "SM-pair kernel"),
    (256, 512, 1024, fp8g.SWAP_OFF | fp8g.SINGLE_SM_TILES, "single-SM kernel, one issuer"),
    (256, 512, 1024, fp8g.SWAP_OFF | fp8g.SINGLE_SM_TILES | fp8g.TILE_N(3), "single-SM kernel, two issuers"),
    (32, 2048, 2048, fp8g.SWAP_ON, "SwapAB kernel, two issuers"),
])
def test_block_scaled_wait_runs_out_then_gpu_still_correct(M, N, K, flags, name):
    """The block-scaled kernels' extra roles (scale-staging warps, a second
    MMA issuer, the scale barriers the loader drains) leave cleanly too."""
    A = synth.normal_fp8((M, K), 611 + M, 0.0, 1.0, synth.E4M3)
    B = synth.normal_fp8((N, K), 612 + N, 0.0, 1.0, synth.E4M3)
    ks = K // 128
    rng = np.random.default_rng(613)
    sfa = rng.integers(124, 131, (1, ks, M)).astype(np.uint8)
    sfb = rng.integers(124, 131, (1, ks, N)).astype(np.uint8)
    Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    sfad, sfbd = torch.from_numpy(sfa).cuda(), torch.from_numpy(sfb).cuda()
    prev = fp8g.fp8g_set_wait_timeout_ns(LIMIT_NS)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        fp8g.fp8_gemm_nt_blockscaled(Ad, Bd, sfad, sfbd, sf_group_k=128, a_dtype=0, b_dtype=0,
                                     flags=flags | fp8g.DEBUG_DROP_FIRST_LOAD)
        st = fp8g.fp8g_get_device_status()
        elapsed = time.perf_counter() - t0
    finally:
        fp8g.fp8g_set_wait_timeout_ns(prev)
    assert st[0] == fp8g.ERR_TIMEOUT, (name, st)
    assert elapsed < 5.0, elapsed
    D = fp8g.fp8_gemm_nt_blockscaled(Ad, Bd, sfad, sfbd, sf_group_k=128, a_dtype=0, b_dtype=0, flags=flags)
    st2 = fp8g.fp8g_get_device_status()
    assert st2[0] == fp8g.OK, st2
    ref, absdot, accb = oracle.gemm_blockscaled(A, B, sfa[0], sfb[0], 128, want_accbound=True)
    ok, rep = oracle.check_bf16(bits(D), ref, absdot, acc_bound=accb)
    assert ok, (name, rep)
