"""fp8_gemm_nt_noalloc, the entry point that allocates no device memory
(for callers whose own allocator must own every device byte, or that cannot
take cudaMalloc's synchronisation).  Its
stream-K scratch is a fixed device array inside the library, shared by every
call, so two calls in a row must both agree with the oracle (and, bit for
bit, with the allocating entry point that runs the same kernel).

A third test checks that the calls take no device memory.

Kept in a file of its own that pytest collects last."""
import ctypes

import numpy as np
import pytest
import torch

import __graft_entry__  # noqa: F401
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    from fp8_tensor_core_gb300 import _lib
    from fp8_tensor_core_gb300 import build as cuda_build
    cuda_build.build()
    torch.cuda.set_device(0)
    return _lib.load()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(64, 7168, 4096), (8, 24576, 1536), (1, 1024, 2048),
                                   (37, 3000, 1040)])
def test_noalloc_matches_the_oracle_twice(lib, M, N, K):
    """Two calls in a row (the second finds the first one's scratch
    contents): each output matches the oracle within the tolerance, and is
    bit-identical to the allocating entry point's output (same kernel, same
    stream-K partition, same K-ordered sums)."""
    A = synth.normal_fp8((M, K), 501 + M, 0.0, 1.0, synth.E4M3)
    B = synth.normal_fp8((N, K), 502 + N, 0.0, 1.0, synth.E4M3)
    Ad = torch.from_numpy(A).cuda()
    Bd = torch.from_numpy(B).cuda()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ref, absdot = oracle.gemm_nt(A, B)
    D_alloc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = lib.fp8_gemm_nt(Ad.data_ptr(), Bd.data_ptr(), D_alloc.data_ptr(), M, N, K, 0, 0, 1, stream)
    assert rc == 0
    for call in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.fp8_gemm_nt_noalloc(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), M, N, K, 0, 0,
                                     stream)
        assert rc == 0, lib.fp8g_status_string(rc)
        torch.cuda.synchronize()
        got = _bits(D)
        ok, rep = oracle.check_bf16(got, ref, absdot)
        assert ok, (call, rep)
        assert np.array_equal(got, _bits(D_alloc)), call
    info = (ctypes.c_int32 * 4)()
    assert lib.fp8g_get_device_status(info, stream) == 0
    assert info[0] == 0, tuple(info)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # M = 256 tokens over N = 65536 weight rows needs ~39 MB of partial tiles
    # (2 x 152 CTAs x 128 x 256 x 4 bytes) plus 16 KB of counters.
    M, N, K = 256, 65536, 16384
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    B = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fp8_gemm_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, 0, 0,
                                   stream) == 3
    assert lib.fp8_gemm_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), 300, 8, 16, 0, 0,
                                   stream) == 3
    torch.cuda.synchronize()
    assert torch.count_nonzero(D).item() == 0


def test_noalloc_takes_no_device_memory(lib):
    """Calls of the no-allocation entry point leave the device's free memory
    unchanged, on a stream no call has used before; the same kind of call
    through fp8_gemm_nt on another new stream does allocate (that stream's
    stream-K scratch), so the check can see an allocation."""
    shapes = [(1, 7168, 4096), (16, 4096, 2048), (64, 7168, 4096), (200, 2048, 1024)]
    bufs = []
    for M, N, K in shapes:
        A = torch.from_numpy(synth.normal_fp8((M, K), 700 + M, 0.0, 1.0, synth.E4M3)).cuda()
        B = torch.from_numpy(synth.normal_fp8((N, K), 701 + N, 0.0, 1.0, synth.E4M3)).cuda()
        bufs.append((A, B, torch.empty((M, N), dtype=torch.bfloat16, device="cuda"), M, N, K))
    warm = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for A, B, D, M, N, K in bufs:   # kernels loaded, device limits looked up
        assert lib.fp8_gemm_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, 0, 0, warm) == 0
    torch.cuda.synchronize()
    s_new = torch.cuda.Stream()
    stream = ctypes.c_void_p(s_new.cuda_stream)
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for A, B, D, M, N, K in bufs:
            assert lib.fp8_gemm_nt_noalloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, 0, 0, stream) == 0
    torch.cuda.synchronize()
    # (1 MB of slack for the device's own bookkeeping; the library's scratch
    # of any call is several MB)
    assert torch.cuda.mem_get_info()[0] >= free0 - (1 << 20)
    # control: the allocating entry point on a new stream (SwapAB, stream-K)
    s_ctl = torch.cuda.Stream()
    A, B, D, M, N, K = bufs[2]
    assert lib.fp8_gemm_nt(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K, 0, 0, 1,
                           ctypes.c_void_p(s_ctl.cuda_stream)) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free0 - (4 << 20)   # 152 x 2 x 128 x 64 FP32 partial tiles
    assert lib.fp8g_release_stream(ctypes.c_void_p(s_ctl.cuda_stream)) == 0
    info = (ctypes.c_int32 * 4)()
    assert lib.fp8g_get_device_status(info, stream) == 0
    assert info[0] == 0, tuple(info)
