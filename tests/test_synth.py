"""The seeded input generator: determinism, slicing, the FP8 encoder against
torch's casts, and the workload distributions."""
import numpy as np
import pytest
import torch

import synth

TORCH_FP8 = {synth.E4M3: torch.float8_e4m3fn, synth.E5M2: torch.float8_e5m2}
MAXV = {synth.E4M3: 448.0, synth.E5M2: 57344.0}
MAXC = {synth.E4M3: 0x7E, synth.E5M2: 0x7B}


def torch_values(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def test_splitmix64_published_values():
    """SplitMix64 seeded with 0: the first outputs of the reference stream."""
    assert synth.splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert synth.splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert synth.splitmix64_at(0, 2) == 0x06C45D188009454F


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_encode_roundtrips_every_finite_code(fmt):
    vals = torch_values(fmt)
    for c in range(256):
        v = vals[c]
        if not np.isfinite(v):
            continue
        got = synth.encode_fp8(v, fmt)
        if v == 0.0:
            assert got == c          # keeps the sign of zero
        else:
            assert got == c, (hex(c), v, hex(got))


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_encode_matches_torch_cast_in_range(fmt):
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 30, 4000),
                        rng.uniform(-2, 2, 4000),
                        rng.normal(0, 1e-3, 2000)]).astype(np.float32)
    x = x[np.abs(x) < MAXV[fmt]]
    ref = torch.from_numpy(x).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    mine = synth.encode_fp8_array(x.astype(np.float64), fmt)
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("fmt", [synth.E4M3, synth.E5M2])
def test_encode_ties_to_even_and_saturates(fmt):
    vals = torch_values(fmt)
    pos = [(c, vals[c]) for c in range(128) if np.isfinite(vals[c])]
    for (c0, v0), (c1, v1) in zip(pos, pos[1:]):
        mid = (v0 + v1) / 2.0                      # exact in double
        want = c0 if c0 % 2 == 0 else c1           # even mantissa code wins
        assert synth.encode_fp8(mid, fmt) == want
        assert synth.encode_fp8(-mid, fmt) == want | 0x80
    for big in (MAXV[fmt] * 1.01, MAXV[fmt] * 100, 1e30, float("inf")):
        assert synth.encode_fp8(big, fmt) == MAXC[fmt]
        assert synth.encode_fp8(-big, fmt) == MAXC[fmt] | 0x80


def test_fill_deterministic_sliceable_thread_independent():
    a = synth.normal_fp8((300, 257), 42, 0.0, 1.0, synth.E4M3, nthreads=1)
    b = synth.normal_fp8((300, 257), 42, 0.0, 1.0, synth.E4M3, nthreads=7)
    assert np.array_equal(a, b)
    tail = synth.rows_fp8("normal", (100, 257), 42, synth.E4M3, row_first=200,
                          std=1.0)
    assert np.array_equal(tail, a[200:])
    c = synth.normal_fp8((300, 257), 43, 0.0, 1.0, synth.E4M3)
    assert not np.array_equal(a, c)


def test_distributions():
    n = 1 << 18
    z = np.array([synth.normal_at(5, i) for i in range(20000)])
    assert abs(z.mean()) < 0.03 and abs(z.std() - 1.0) < 0.03
    u = synth.uniform_fp8((n,), 9, -2.0, 2.0, synth.E4M3)
    v = torch.from_numpy(u).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert v.min() >= -2.0 and v.max() <= 2.0 and abs(v.mean()) < 0.02
    m = synth.uniform_int(100000, 3, 0, 32)
    assert m.min() == 0 and m.max() == 32
    counts = np.bincount(m, minlength=33)
    assert counts.min() > 2500                    # ~3030 each
