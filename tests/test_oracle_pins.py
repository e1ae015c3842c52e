"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- torch's float8 / bfloat16 conversions, exact rational
brute force, closed forms of structured products, printed fixtures -- so that
a dropped term, a wrong sign or index, or a transposed operand fails here."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMTS = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def torch_decode_all(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def torch_decode(codes: np.ndarray, fmt) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return t.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


# ---- FP8 decode --------------------------------------------------------------

@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_all_codes_match_torch(fmt):
    mine = oracle.decode_table(fmt)
    ref = torch_decode_all(fmt)
    nan_m, nan_r = np.isnan(mine), np.isnan(ref)
    assert np.array_equal(nan_m, nan_r)
    assert np.array_equal(mine[~nan_m], ref[~nan_r])
    # signed zeros: 0x80 is -0 in both formats
    assert math.copysign(1.0, mine[0x80]) == -1.0
    for c in range(256):
        assert oracle.decode_fp8(c, fmt) == mine[c] or (np.isnan(mine[c]))


def _golden_points():
    pts = []
    with open(os.path.join(GOLDEN, "fp8_format_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            fmt, code, val = line.split()
            pts.append((FMTS[fmt], int(code, 16), val))
    return pts


@pytest.mark.parametrize("fmt,code,val", _golden_points())
def test_decode_golden_points(fmt, code, val):
    got = oracle.decode_fp8(code, fmt)
    if val == "nan":
        assert math.isnan(got)
    elif val in ("inf", "-inf"):
        assert got == float(val)
    elif val == "-0":
        assert got == 0.0 and math.copysign(1.0, got) == -1.0
    else:
        assert Fraction(got) == Fraction(val)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_structure(fmt):
    """Positive finite codes are strictly increasing in code order, the
    negative half mirrors the positive half, and NaN counts match the
    format (E4M3: 2 NaN codes, no inf; E5M2: 6 NaN codes, 2 inf)."""
    t = oracle.decode_table(fmt)
    pos = t[:128]
    fin = pos[np.isfinite(pos)]
    assert np.all(np.diff(fin) > 0)
    for c in range(128):
        if np.isnan(t[c]):
            assert np.isnan(t[c | 0x80])
        else:
            assert t[c | 0x80] == -t[c]
    n_nan = int(np.isnan(t).sum())
    n_inf = int(np.isinf(t).sum())
    assert (n_nan, n_inf) == ((2, 0) if fmt == oracle.E4M3 else (6, 2))


# ---- BF16 rounding -----------------------------------------------------------

def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add values right at and around BF16 midpoints
    mids = (rng.integers(0, 2**16, 5000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    near = np.concatenate([mids, mids + 1, mids - 1]).astype(np.uint32).view(np.float32)
    near = near[np.isfinite(near)]
    vals = np.concatenate([f, near]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = oracle.round_bf16_array(vals.astype(np.float64))
    # torch maps NaN to a canonical NaN too; none here (finite inputs only)
    assert np.array_equal(mine, ref)


def test_round_bf16_ties_and_specials_exact():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties to even -> 1.0
    assert oracle.round_bf16(1.0 + 2**-8) == 0x3F80
    # 1 + 3*2^-8 is the midpoint of 1+2^-7 (odd) and 1+2^-6 (even) -> up
    assert oracle.round_bf16(1.0 + 3 * 2**-8) == 0x3F82
    # just above a tie rounds up (needs more than float32 precision)
    assert oracle.round_bf16(1.0 + 2**-8 + 2**-40) == 0x3F81
    assert oracle.round_bf16(-(1.0 + 2**-8 + 2**-40)) == 0xBF81
    assert oracle.round_bf16(0.0) == 0x0000
    assert oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(float("inf")) == 0x7F80
    assert oracle.round_bf16(3.5e38) == 0x7F80           # overflow
    assert oracle.round_bf16(2.0**-133) == 0x0001        # smallest subnormal
    assert oracle.round_bf16(2.0**-134) == 0x0000        # tie to even (zero)
    assert oracle.round_bf16(3 * 2.0**-134) == 0x0002    # tie to even (2)
    assert oracle.round_bf16(255.5) == oracle.round_bf16(256.0) == 0x4380
    for h in (0x3F80, 0x4000, 0x0001, 0x7F7F, 0x8001):
        assert oracle.round_bf16(oracle.bf16_to_double(h)) == h


def _rne_fraction_to_bf16(x: Fraction) -> int:
    """Independent exact rounding of a rational to BF16 by search over the
    representable neighbours (no floating point involved)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    # candidate codes: find k with 2^k <= a < 2^(k+1)
    k = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** k > a:
        k -= 1
    while Fraction(2) ** (k + 1) <= a:
        k += 1
    k = max(k, -126)
    sp = Fraction(2) ** (k - 7)
    lo = (a / sp).__floor__()
    cands = [lo, lo + 1]
    best = min(cands, key=lambda c: (abs(a - c * sp), c % 2))
    val = best * sp
    # encode val exactly
    num = val / Fraction(2) ** -133
    if num < 128:
        return sign | int(num)
    e = val.numerator.bit_length() - val.denominator.bit_length()
    while Fraction(2) ** e > val:
        e -= 1
    while Fraction(2) ** (e + 1) <= val:
        e += 1
    m = val / Fraction(2) ** (e - 7) - 128
    return sign | ((e + 127) << 7) | int(m)


# ---- the contraction -----------------------------------------------------------

def _rand_codes(shape, seed, fmt, std=1.0):
    return synth.normal_fp8(shape, seed, 0.0, std, fmt)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (2, 3, 16), (3, 2, 17),
                                   (16, 17, 32), (17, 16, 3), (5, 7, 32)])
@pytest.mark.parametrize("fa,fb", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_exact_rational_bruteforce(M, N, K, fa, fb):
    """Exact rational triple loop (values from torch's float8 decode) rounded
    exactly to BF16 must equal the oracle bit for bit."""
    A = _rand_codes((M, K), 11 + M * 7 + K, fa, std=4.0)
    B = _rand_codes((N, K), 97 + N * 5 + K, fb, std=4.0)
    da, db = torch_decode(A, fa), torch_decode(B, fb)
    D, absdot, exact = oracle.gemm_nt(A, B, fa, fb, want_exact=True)
    for m in range(M):
        for n in range(N):
            s = sum((Fraction(da[m, k]) * Fraction(db[n, k]) for k in range(K)),
                    Fraction(0))
            assert D[m, n] == _rne_fraction_to_bf16(s), (m, n)
            assert Fraction(exact[m, n]) == s          # small K: double exact
            assert absdot[m, n] == float(sum(abs(Fraction(da[m, k]) * Fraction(db[n, k]))
                                             for k in range(K)))


@pytest.mark.parametrize("fa,fb", [(0, 0), (0, 1), (1, 1)])
def test_gemm_matches_numpy_matmul(fa, fb):
    """Against a library routine: numpy float64 matmul of torch-decoded
    operands; agreement to double rounding noise, and BF16 codes within one
    ulp (double rounding near ties can move the last bit)."""
    M, N, K = 33, 47, 1000
    A = _rand_codes((M, K), 5, fa)
    B = _rand_codes((N, K), 6, fb)
    D, absdot, exact = oracle.gemm_nt(A, B, fa, fb, want_exact=True)
    ref = torch_decode(A, fa) @ torch_decode(B, fb).T
    assert np.all(np.abs(exact - ref) <= 1e-12 * absdot + 1e-300)
    ref_bits = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    d = np.abs(D.astype(np.int64) - ref_bits.astype(np.int64))
    assert d.max() <= 1
    assert np.mean(d == 0) > 0.99


@pytest.mark.parametrize("fmt,one", [(oracle.E4M3, 0x38), (oracle.E5M2, 0x3C)])
def test_gemm_identity_gives_transpose(fmt, one):
    """A = I (M = K) gives D = B^T exactly, since every FP8 value is exact in
    BF16; a transposed operand or a wrong index fails this (B is random and
    not symmetric)."""
    K, N = 48, 40
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = one
    B = _rand_codes((N, K), 77, fmt)
    D, _ = oracle.gemm_nt(A, B, fmt, fmt)
    ref = torch.from_numpy(torch_decode(B, fmt).T.copy()).to(torch.bfloat16)
    assert np.array_equal(D, ref.view(torch.int16).numpy().view(np.uint16))


def test_gemm_permutation_permutes_rows():
    K, N = 32, 24
    perm = np.random.default_rng(3).permutation(K)
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), perm] = 0x38          # row m picks k = perm[m]
    B = _rand_codes((N, K), 78, oracle.E4M3)
    D, _ = oracle.gemm_nt(A, B)
    Dt, _ = oracle.gemm_nt(np.eye(K, dtype=np.uint8) * 0x38, B)
    assert np.array_equal(D, Dt[perm])


def test_gemm_single_nonzero_k_is_exact_product():
    fa, fb = oracle.E4M3, oracle.E5M2
    K = 64
    for kk, ca, cb in [(0, 0x38, 0x40), (17, 0x7E, 0x3C), (63, 0xB9, 0x3D), (5, 0x01, 0x04)]:
        A = np.zeros((1, K), np.uint8)
        B = np.zeros((1, K), np.uint8)
        A[0, kk], B[0, kk] = ca, cb
        D, _, ex = oracle.gemm_nt(A, B, fa, fb, want_exact=True)
        p = oracle.decode_fp8(ca, fa) * oracle.decode_fp8(cb, fb)
        assert ex[0, 0] == p
        assert D[0, 0] == oracle.round_bf16(p)


def test_gemm_integer_valued_products_exact():
    """Entries in {-2,-1,0,1,2} (exact in both formats) with |sum| <= 256 give
    exact BF16 results equal to an integer matmul."""
    rng = np.random.default_rng(9)
    vals = np.array([-2, -1, 0, 1, 2])
    enc = {oracle.E4M3: {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40},
           oracle.E5M2: {-2: 0xC0, -1: 0xBC, 0: 0x00, 1: 0x3C, 2: 0x40}}
    M, N, K = 20, 30, 64
    ia = rng.choice(vals, (M, K))
    ib = rng.choice(vals, (N, K))
    for fa, fb in [(0, 0), (0, 1), (1, 1)]:
        A = np.vectorize(enc[fa].get)(ia).astype(np.uint8)
        B = np.vectorize(enc[fb].get)(ib).astype(np.uint8)
        D, _ = oracle.gemm_nt(A, B, fa, fb)
        ref = ia.astype(np.int64) @ ib.T.astype(np.int64)
        assert np.abs(ref).max() <= 256
        got = oracle.bf16_bits_to_f64(D)
        assert np.array_equal(got, ref.astype(np.float64))


@pytest.mark.parametrize("K", [1, 16, 128, 255, 256])
def test_gemm_all_ones_is_K(K):
    A = np.full((3, K), 0x38, np.uint8)
    B = np.full((5, K), 0x38, np.uint8)
    D, absdot = oracle.gemm_nt(A, B)
    assert np.all(oracle.bf16_bits_to_f64(D) == K)
    assert np.all(absdot == K)


def test_gemm_entries_match_full():
    A = _rand_codes((40, 200), 1, oracle.E4M3)
    B = _rand_codes((30, 200), 2, oracle.E5M2)
    D, absdot = oracle.gemm_nt(A, B, 0, 1)
    ms = np.array([0, 39, 7, 20, 13])
    ns = np.array([0, 29, 11, 3, 29])
    d, ad, _ = oracle.gemm_nt_entries(A, B, ms, ns, 0, 1)
    assert np.array_equal(d, D[ms, ns])
    assert np.array_equal(ad, absdot[ms, ns])


def test_gemm_threads_do_not_change_results():
    A = _rand_codes((64, 300), 3, oracle.E4M3)
    B = _rand_codes((50, 300), 4, oracle.E4M3)
    D1, a1 = oracle.gemm_nt(A, B, nthreads=1)
    D8, a8 = oracle.gemm_nt(A, B, nthreads=8)
    assert np.array_equal(D1, D8) and np.array_equal(a1, a8)


# ---- masked grouped --------------------------------------------------------------

def test_grouped_masked_rows_and_untouched_padding():
    G, M_max, N, K = 5, 24, 16, 48
    A = _rand_codes((G, M_max, K), 21, oracle.E4M3)
    B = _rand_codes((G, N, K), 22, oracle.E4M3)
    mm = np.array([0, 1, 24, 7, 16], np.int32)
    D0 = synth.u16_pattern((G, M_max, N), 23)
    D, absdot = oracle.gemm_grouped_masked(A, B, mm, D0)
    for g in range(G):
        m = mm[g]
        ref, _ = oracle.gemm_nt(A[g, :m], B[g])
        assert np.array_equal(D[g, :m], ref)
        assert np.array_equal(D[g, m:], D0[g, m:])      # never written
        assert np.all(absdot[g, m:] == 0)


def test_grouped_masked_nan_padding_does_not_leak():
    G, M_max, N, K = 2, 16, 8, 32
    A = _rand_codes((G, M_max, K), 31, oracle.E4M3)
    B = _rand_codes((G, N, K), 32, oracle.E4M3)
    mm = np.array([5, 9], np.int32)
    A2 = A.copy()
    for g in range(G):
        A2[g, mm[g]:] = 0x7F                               # NaN codes in padding
    D0 = np.zeros((G, M_max, N), np.uint16)
    Da, _ = oracle.gemm_grouped_masked(A, B, mm, D0)
    Db, _ = oracle.gemm_grouped_masked(A2, B, mm, D0)
    assert np.array_equal(Da, Db)


# ---- acceptance rule -----------------------------------------------------------

def test_check_bf16_rule():
    ref = np.array([0x3F80, 0x3F80, 0x3F80, 0x0000, 0x3F80], np.uint16)   # 1.0 ...
    absdot = np.array([1.0, 1.0, 1.0, 1.0, 1e6])
    one_ulp = np.array([0x3F81, 0x3F7F, 0x3F80, 0x0000, 0x3F83], np.uint16)
    ok, rep = oracle.check_bf16(one_ulp, ref, absdot)
    assert ok, rep                                   # last one: 3 ulp < 1e-6*1e6
    two_ulp = np.array([0x3F82], np.uint16)
    ok, _ = oracle.check_bf16(two_ulp, ref[:1], absdot[:1])
    assert not ok
    ok, _ = oracle.check_bf16(np.array([0x7FC0], np.uint16), ref[:1], absdot[:1])
    assert not ok                                    # NaN never passes
    assert oracle.ulp_bf16(np.array([0x3F80]))[0] == 2.0**-7
    assert oracle.ulp_bf16(np.array([0x0000]))[0] == 0.0


def test_planted_transpose_mistake_is_caught():
    """A plausible oracle bug (B indexed as [k, n] instead of [n, k]) must be
    caught by the identity pin: emulate it on the CPU and check the pin's
    comparison fails."""
    K = 32
    A = np.eye(K, dtype=np.uint8) * 0x38
    B = _rand_codes((K, K), 79, oracle.E4M3)
    wrong, _ = oracle.gemm_nt(A, np.ascontiguousarray(B.T))    # planted bug
    ref = torch.from_numpy(torch_decode(B, 0).T.copy()).to(torch.bfloat16)
    assert not np.array_equal(wrong, ref.view(torch.int16).numpy().view(np.uint16))


def test_planted_sign_mistake_is_caught():
    """Negating a decoded term (a sign error) is caught by the rational brute
    force: the results differ on random data."""
    A = _rand_codes((4, 16), 81, oracle.E4M3)
    B = _rand_codes((4, 16), 82, oracle.E4M3)
    D, _ = oracle.gemm_nt(A, B)
    Dneg, _ = oracle.gemm_nt(A ^ 0x80, B)           # planted: flipped sign bits
    assert not np.array_equal(D, Dneg)


# ---- scaled variants --------------------------------------------------------------

def test_scaled_power_of_two_scales_shift_exponents_exactly():
    """Per-row/per-column scales 2^e multiply the exact sum exactly, so the
    BF16 result is the unscaled one with its exponent shifted."""
    A = _rand_codes((24, 96), 201, oracle.E4M3)
    B = _rand_codes((40, 96), 202, oracle.E4M3)
    ea = np.random.default_rng(1).integers(-6, 7, 24)
    eb = np.random.default_rng(2).integers(-6, 7, 40)
    sa = np.ldexp(1.0, ea).astype(np.float32)
    sb = np.ldexp(1.0, eb).astype(np.float32)
    D, absdot = oracle.gemm_nt_scaled(A, B, sa, sb)
    D0, absdot0 = oracle.gemm_nt(A, B)
    want = oracle.bf16_bits_to_f64(D0) * np.ldexp(1.0, ea[:, None] + eb[None, :])
    assert np.array_equal(oracle.bf16_bits_to_f64(D), want)
    assert np.allclose(absdot, absdot0 * np.ldexp(1.0, ea[:, None] + eb[None, :]), rtol=0, atol=0)


def test_scaled_unit_and_per_tensor_scales():
    A = _rand_codes((16, 64), 203, oracle.E5M2)
    B = _rand_codes((24, 64), 204, oracle.E4M3)
    D0, _ = oracle.gemm_nt(A, B, 1, 0)
    D1, _ = oracle.gemm_nt_scaled(A, B, np.ones(1, np.float32), np.ones(24, np.float32), 1, 0)
    assert np.array_equal(D0, D1)
    Dt, _ = oracle.gemm_nt_scaled(A, B, np.array([0.375], np.float32), np.array([-3.0], np.float32), 1, 0)
    Dr, _ = oracle.gemm_nt_scaled(A, B, np.full(16, 0.375, np.float32), np.full(24, -3.0, np.float32), 1, 0)
    assert np.array_equal(Dt, Dr)


def test_scaled_matches_numpy_reference():
    """Against numpy float64 products of torch-decoded operands and the
    scales; BF16 codes within one ulp (numpy's path rounds through float32)."""
    A = _rand_codes((37, 200), 205, oracle.E4M3)
    B = _rand_codes((29, 200), 206, oracle.E4M3)
    rng = np.random.default_rng(3)
    sa = rng.uniform(0.01, 4.0, 37).astype(np.float32)
    sb = rng.uniform(-2.0, 2.0, 29).astype(np.float32)
    D, _ = oracle.gemm_nt_scaled(A, B, sa, sb)
    ref = (sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
           * (torch_decode(A, 0) @ torch_decode(B, 0).T))
    ref_bits = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    d = np.abs(D.astype(np.int64) - ref_bits.astype(np.int64))
    assert d.max() <= 1 and np.mean(d == 0) > 0.98


def test_grouped_scaled_per_group_and_per_row():
    G, M_max, N, K = 4, 16, 24, 64
    A = _rand_codes((G, M_max, K), 207, oracle.E4M3)
    B = _rand_codes((G, N, K), 208, oracle.E4M3)
    mm = np.array([3, 0, 16, 9], np.int32)
    sa_g = np.array([0.5, 2.0, 1.25, -1.0], np.float32)
    sb_gn = np.random.default_rng(4).uniform(0.5, 2.0, G * N).astype(np.float32)
    D0 = synth.u16_pattern((G, M_max, N), 209)
    D, _ = oracle.gemm_grouped_masked_scaled(A, B, mm, sa_g, sb_gn, D0)
    for g in range(G):
        m = mm[g]
        ref, _ = oracle.gemm_nt_scaled(A[g, :m], B[g], sa_g[g:g + 1], sb_gn[g * N:(g + 1) * N])
        assert np.array_equal(D[g, :m], ref)
        assert np.array_equal(D[g, m:], D0[g, m:])
    sa_r = np.random.default_rng(5).uniform(0.5, 2.0, G * M_max).astype(np.float32)
    D2, _ = oracle.gemm_grouped_masked_scaled(A, B, mm, sa_r, sa_g, D0)
    g = 2
    ref, _ = oracle.gemm_nt_scaled(A[g], B[g], sa_r[g * M_max:(g + 1) * M_max], sa_g[g:g + 1])
    assert np.array_equal(D2[g], ref)


# ---- block-scaled variant -----------------------------------------------------------

def _ue8m0(shape, seed, lo=124, hi=130):
    return np.random.default_rng(seed).integers(lo, hi + 1, shape).astype(np.uint8)


@pytest.mark.parametrize("M,N,K,gran", [(3, 4, 40, 32), (5, 2, 130, 128), (2, 3, 96, 32), (4, 4, 17, 128)])
def test_blockscaled_exact_rational_bruteforce(M, N, K, gran):
    """Exact rational sum of a_k b_k 2^(ea-127) 2^(eb-127) over k, rounded
    exactly to BF16, equals the oracle bit for bit."""
    A = _rand_codes((M, K), 301 + K, 0)
    B = _rand_codes((N, K), 302 + K, 1)
    KS = -(-K // gran)
    sfa = _ue8m0((KS, M + 3), 303 + K)             # ld > M: padding bytes unused
    sfb = _ue8m0((KS, N), 304 + K)
    D, absdot = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, fa=0, fb=1)
    da, db = torch_decode(A, 0), torch_decode(B, 1)
    for m in range(M):
        for n in range(N):
            terms = [Fraction(da[m, k]) * Fraction(db[n, k])
                     * Fraction(2) ** (int(sfa[k // gran, m]) - 127)
                     * Fraction(2) ** (int(sfb[k // gran, n]) - 127) for k in range(K)]
            assert D[m, n] == _rne_fraction_to_bf16(sum(terms, Fraction(0))), (m, n)
            assert absdot[m, n] == float(sum(abs(t) for t in terms))


@pytest.mark.parametrize("K,slices", [(128, [32, 64, 96, 128]), (80, [32, 64, 80]), (32, [32]), (16, [16])])
def test_blockscaled_accbound_closed_form(K, slices):
    """All-ones operands with unit scales: the running sum after each
    32-element slice is its length, so the bound is 2^-23 times the sum of
    the slice ends (a shorter last slice counted once)."""
    A = np.full((2, K), 0x38, np.uint8)        # E4M3 1.0
    B = np.full((3, K), 0x38, np.uint8)
    KS = -(-K // 32)
    one = np.full((KS, 16), 127, np.uint8)
    D, absdot, accb = oracle.gemm_blockscaled(A, B, one, one, 32, want_accbound=True)
    assert np.all(absdot == K)
    assert np.all(accb == math.ldexp(sum(slices), -23))


def _fp32_accumulate(parts, mode):
    """A float32 accumulator that adds each exact slice sum with one rounding,
    to nearest even or toward zero."""
    acc = np.zeros(parts.shape[:-1], np.float64)
    for i in range(parts.shape[-1]):
        x = acc + parts[..., i]                    # exact: both terms are float32 / short sums
        r = x.astype(np.float32).astype(np.float64)
        if mode == "rz":
            over = np.abs(r) > np.abs(x)
            r = np.where(over, np.nextafter(r.astype(np.float32), np.float32(0)).astype(np.float64), r)
        acc = r
    return acc


@pytest.mark.parametrize("gran", [32, 128])
def test_blockscaled_accbound_bounds_fp32_accumulation(gran):
    """The bound holds for an FP32 accumulator that adds each 32-element
    slice's exact sum with one rounding -- toward zero (the worst direction)
    or to nearest -- on data whose K groups differ by up to 2^28 in scale,
    and never exceeds the crude bound n * 2^-23 * sum |a b| that ignores the
    running sums."""
    M, N, K = 12, 20, 1024
    A = _rand_codes((M, K), 331, 0)
    B = _rand_codes((N, K), 332, 0)
    KS = -(-K // gran)
    sfa = _ue8m0((KS, M + 4), 333, 113, 141)
    sfb = _ue8m0((KS, N + 12), 334, 113, 141)
    D, absdot, exact, accb = oracle.gemm_blockscaled(A, B, sfa, sfb, gran, want_exact=True, want_accbound=True)
    da, db = torch_decode(A, 0), torch_decode(B, 0)
    g = np.arange(K) // gran
    sa = np.ldexp(1.0, sfa[g, :M].T.astype(np.int64) - 127)          # [M, K]
    sb = np.ldexp(1.0, sfb[g, :N].T.astype(np.int64) - 127)          # [N, K]
    prod = (da * sa)[:, None, :] * (db * sb)[None, :, :]             # [M, N, K], exact
    parts = prod.reshape(M, N, K // 32, 32).sum(axis=-1)             # exact: one scale pair per slice
    worst = 0.0
    for mode in ("rz", "rn"):
        err = np.abs(_fp32_accumulate(parts, mode) - exact)
        assert np.all(err <= accb), mode
        worst = max(worst, float((err / accb).max()))
    assert worst > 0.05                              # the bound is not vacuous on this data
    assert np.all(accb <= (K // 32) * 2.0 ** -23 * absdot * (1 + 1e-12))


@pytest.mark.parametrize("gran", [32, 128])
def test_blockscaled_unit_scales_equal_unscaled(gran):
    A = _rand_codes((20, 200), 311, 0)
    B = _rand_codes((12, 200), 312, 0)
    KS = -(-200 // gran)
    D, _ = oracle.gemm_blockscaled(A, B, np.full((KS, 20), 127, np.uint8), np.full((KS, 16), 127, np.uint8), gran)
    D0, _ = oracle.gemm_nt(A, B)
    assert np.array_equal(D, D0)


def test_blockscaled_constant_row_scales_shift_exponents():
    """Scales constant along K act as per-row / per-column powers of two:
    the unscaled result with its exponent shifted, exactly."""
    A = _rand_codes((24, 384), 313, 0)
    B = _rand_codes((16, 384), 314, 0)
    ea = np.random.default_rng(6).integers(110, 145, 24)
    eb = np.random.default_rng(7).integers(110, 145, 16)
    sfa = np.tile(ea.astype(np.uint8), (3, 1))
    sfb = np.tile(eb.astype(np.uint8), (3, 1))
    D, _ = oracle.gemm_blockscaled(A, B, sfa, sfb, 128)
    D0, _ = oracle.gemm_nt(A, B)
    want = oracle.bf16_bits_to_f64(D0) * np.ldexp(1.0, (ea - 127)[:, None] + (eb - 127)[None, :])
    assert np.array_equal(oracle.bf16_bits_to_f64(D), want)


@pytest.mark.parametrize("gran", [32, 128])
def test_blockscaled_isolates_each_k_group(gran):
    """Scale 1 on one K group and 2^-127 on the others leaves (up to a
    leak below 2^-90) the unscaled product of that group's K slice alone --
    so a transposed or mis-strided scale index fails here."""
    M, N, K = 9, 7, 200
    A = _rand_codes((M, K), 315, 0)
    B = _rand_codes((N, K), 316, 0)
    KS = -(-K // gran)
    for j in range(KS):
        sfa = np.zeros((KS, M), np.uint8)
        sfa[j] = 127
        sfb = np.full((KS, N), 127, np.uint8)
        D, _ = oracle.gemm_blockscaled(A, B, sfa, sfb, gran)
        lo, hi = j * gran, min(K, (j + 1) * gran)
        _, _, exact = oracle.gemm_nt(A[:, lo:hi].copy(), B[:, lo:hi].copy(), want_exact=True)
        got = oracle.bf16_bits_to_f64(D)
        ref = oracle.bf16_bits_to_f64(np.array([[oracle.round_bf16(v) for v in r] for r in exact], np.uint16))
        assert np.all(np.abs(got - ref) <= 2.0 ** -90), j


def test_blockscaled_gran32_replicated_equals_gran128():
    A = _rand_codes((10, 300), 317, 0)
    B = _rand_codes((6, 300), 318, 1)
    s128a, s128b = _ue8m0((3, 10), 319), _ue8m0((3, 6), 320)
    s32a = np.repeat(s128a, 4, axis=0)[:10]        # ceil(300/32) = 10 groups
    s32b = np.repeat(s128b, 4, axis=0)[:10]
    D128, _ = oracle.gemm_blockscaled(A, B, s128a, s128b, 128, fb=1)
    D32, _ = oracle.gemm_blockscaled(A, B, s32a, s32b, 32, fb=1)
    assert np.array_equal(D128, D32)


def test_blockscaled_nan_code_poisons_its_rows_only():
    A = _rand_codes((6, 256), 321, 0)
    B = _rand_codes((5, 256), 322, 0)
    sfa = np.full((2, 6), 127, np.uint8)
    sfb = np.full((2, 5), 127, np.uint8)
    sfa[1, 4] = 255
    D, _ = oracle.gemm_blockscaled(A, B, sfa, sfb, 128)
    vals = oracle.bf16_bits_to_f64(D)
    assert np.all(np.isnan(vals[4])) and not np.any(np.isnan(np.delete(vals, 4, axis=0)))


def test_blockscaled_grouped_matches_dense_and_keeps_padding():
    G, M_max, N, K = 3, 8, 10, 160
    A = _rand_codes((G, M_max, K), 323, 0)
    B = _rand_codes((G, N, K), 324, 0)
    sfa = _ue8m0((G, 2, 16), 325)
    sfb = _ue8m0((G, 2, N), 326)
    mm = np.array([5, 0, 8], np.int32)
    D0 = synth.u16_pattern((G, M_max, N), 327)
    D, _ = oracle.gemm_blockscaled(A, B, sfa, sfb, 128, masked_m=mm, D_init=D0)
    for g in range(G):
        ref, _ = oracle.gemm_blockscaled(A[g], B[g], sfa[g], sfb[g], 128)
        m = mm[g]
        assert np.array_equal(D[g, :m], ref[:m])
        assert np.array_equal(D[g, m:], D0[g, m:])


# ---- directed BF16 rounding and the fused epilogue ------------------------------------

def _round_fraction_to_bf16(x: Fraction, mode: int) -> int:
    """Exact directed rounding of a rational to BF16 by choosing between the
    two representable neighbours (no floating point)."""
    if mode == 0:
        return _rne_fraction_to_bf16(x)
    if x == 0:
        return 0
    neg = x < 0
    a = abs(x)
    k = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** k > a:
        k -= 1
    while Fraction(2) ** (k + 1) <= a:
        k += 1
    k = max(k, -126)
    sp = Fraction(2) ** (k - 7)
    lo = (a / sp).__floor__()
    away = (mode == 2 and not neg) or (mode == 3 and neg)
    mag = lo + 1 if (away and lo * sp != a) else lo
    val = mag * sp
    biggest = (2 - Fraction(1, 128)) * Fraction(2) ** 127
    if val > biggest:
        return (0x8000 if neg else 0) | (0x7F80 if away else 0x7F7F)
    code = _rne_fraction_to_bf16(val)          # val is representable: exact encode
    return code | (0x8000 if neg else 0)


def _specials():
    vals = [1.0, -1.0, 1.5, 3.0e38, -3.3e38, 3.4e38, 1e-40, -1e-40, 2.0 ** -133, 2.0 ** -134 * 3,
            9.2e-39, 1.0 + 2.0 ** -8, 1.0 + 2.0 ** -9, -(1.0 + 2.0 ** -7 + 2.0 ** -30), 7.0e-45]
    rng = np.random.default_rng(11)
    vals += list(rng.standard_normal(300) * np.exp2(rng.uniform(-140, 130, 300)))
    return vals


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_round_bf16_modes_exact_rational(mode):
    for v in _specials():
        assert oracle.round_bf16_mode(v, mode) == _round_fraction_to_bf16(Fraction(v), mode), (v, mode)


def test_round_bf16_modes_float32_bit_rule():
    """For a float32 input BF16 is its top half: toward zero drops the low 16
    bits; away from zero in the value's direction adds one unit when any
    dropped bit is set (a carry may reach infinity)."""
    rng = np.random.default_rng(12)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    keep = np.isfinite(f)
    bits, f = bits[keep], f[keep]
    top = (bits >> 16).astype(np.uint16)
    low = (bits & 0xFFFF) != 0
    neg = (bits >> 31) == 1
    for i in range(0, bits.size, 37):
        v = float(f[i])
        assert oracle.round_bf16_mode(v, 1) == top[i]
        up = top[i] + (1 if (low[i] and not neg[i]) else 0)
        dn = top[i] + (1 if (low[i] and neg[i]) else 0)
        assert oracle.round_bf16_mode(v, 2) == up, v
        assert oracle.round_bf16_mode(v, 3) == dn, v


def test_round_bf16_modes_order_and_symmetry():
    for v in _specials():
        rd = oracle.bf16_to_double(oracle.round_bf16_mode(v, 3))
        ru = oracle.bf16_to_double(oracle.round_bf16_mode(v, 2))
        rn = oracle.bf16_to_double(oracle.round_bf16_mode(v, 0))
        rz = oracle.bf16_to_double(oracle.round_bf16_mode(v, 1))
        assert rd <= v <= ru and rn in (rd, ru)
        assert rz == (rd if v >= 0 else ru)
        assert oracle.round_bf16_mode(-v, 3) == oracle.round_bf16_mode(v, 2) ^ 0x8000


def test_epilogue_identity_bias_c_alpha():
    A = _rand_codes((12, 96), 401, 0)
    B = _rand_codes((20, 96), 402, 0)
    D0, absd, S = oracle.gemm_nt(A, B, want_exact=True)
    D1, _ = oracle.epilogue(S, absd)                              # alpha 1, nothing else
    assert np.array_equal(D0, D1)
    bias = np.random.default_rng(13).standard_normal(20).astype(np.float32)
    Db, _ = oracle.epilogue(np.zeros_like(S), np.zeros_like(S), bias=bias)
    assert np.array_equal(Db, np.tile(oracle.round_bf16_array(bias.astype(np.float64)), (12, 1)))
    C = synth.u16_pattern((12, 20), 403) & 0x7F7F                 # finite codes of both signs
    for mode in range(4):
        Dc, _ = oracle.epilogue(S, absd, alpha=0.0, beta=1.0, C=C, mode=mode)
        assert np.array_equal(oracle.bf16_bits_to_f64(Dc), oracle.bf16_bits_to_f64(C)), mode
    D4, _ = oracle.epilogue(S, absd, alpha=4.0)
    assert np.array_equal(oracle.bf16_bits_to_f64(D4), 4 * oracle.bf16_bits_to_f64(D0))


def test_epilogue_relu_and_modes_bracket():
    A = _rand_codes((16, 64), 404, 0)
    B = _rand_codes((16, 64), 405, 1)
    _, absd, S = oracle.gemm_nt(A, B, 0, 1, want_exact=True)
    bias = np.linspace(-3, 3, 16).astype(np.float32)
    C = synth.u16_pattern((16, 16), 406) & 0x3FFF
    plain, _ = oracle.epilogue(S, absd, 0.5, -2.0, C, bias)
    relu, _ = oracle.epilogue(S, absd, 0.5, -2.0, C, bias, relu=True)
    pv, rv = oracle.bf16_bits_to_f64(plain), oracle.bf16_bits_to_f64(relu)
    assert np.array_equal(rv, np.maximum(pv, 0.0))
    v = 0.5 * S - 2.0 * oracle.bf16_bits_to_f64(C) + bias[None, :].astype(np.float64)
    dn = oracle.bf16_bits_to_f64(oracle.epilogue(S, absd, 0.5, -2.0, C, bias, mode=3)[0])
    up = oracle.bf16_bits_to_f64(oracle.epilogue(S, absd, 0.5, -2.0, C, bias, mode=2)[0])
    assert np.all(dn <= v) and np.all(v <= up)
    assert np.all((pv == dn) | (pv == up))


def test_epilogue_grouped_masked_rows_untouched():
    G, M_max, N = 3, 5, 8
    S = np.random.default_rng(14).standard_normal((G, M_max, N))
    D0 = synth.u16_pattern((G, M_max, N), 407)
    mm = np.array([2, 0, 5], np.int32)
    bias = np.random.default_rng(15).standard_normal((G, N)).astype(np.float32)
    D, _ = oracle.epilogue(S, np.abs(S), bias=bias, masked_m=mm, D_init=D0)
    for g in range(G):
        assert np.array_equal(D[g, mm[g]:], D0[g, mm[g]:])
        want = oracle.round_bf16_array(S[g, :mm[g]] + bias[g][None, :].astype(np.float64))
        assert np.array_equal(D[g, :mm[g]], want)


# ---- contiguous grouped layout -------------------------------------------------------

def test_contiguous_equals_per_group_dense_and_keeps_other_rows():
    G, N, K = 4, 24, 80
    off = np.array([3, 3, 10, 27, 40], np.int32)          # an empty group, rows 0-2 and 40+ outside
    M_total = 45
    A = _rand_codes((M_total, K), 501, 0)
    B = _rand_codes((G, N, K), 502, 1)
    D0 = synth.u16_pattern((M_total, N), 503)
    D, absd = oracle.gemm_grouped_contiguous(A, B, off, D0, 0, 1)
    for g in range(G):
        r0, r1 = off[g], off[g + 1]
        if r1 > r0:
            ref, ad = oracle.gemm_nt(A[r0:r1], B[g], 0, 1)
            assert np.array_equal(D[r0:r1], ref) and np.array_equal(absd[r0:r1], ad)
    assert np.array_equal(D[:3], D0[:3]) and np.array_equal(D[40:], D0[40:])


def test_contiguous_equals_masked_layout_rows():
    """Packing each masked group's valid rows back to back gives the same
    products as the masked layout (the two layouts hold the same problem)."""
    G, M_max, N, K = 5, 12, 16, 64
    A = _rand_codes((G, M_max, K), 504, 0)
    B = _rand_codes((G, N, K), 505, 0)
    mm = np.array([4, 0, 12, 7, 1], np.int32)
    Dm, _ = oracle.gemm_grouped_masked(A, B, mm, np.zeros((G, M_max, N), np.uint16))
    off = np.concatenate([[0], np.cumsum(mm)]).astype(np.int32)
    Ac = np.concatenate([A[g, :mm[g]] for g in range(G)])
    Dc, _ = oracle.gemm_grouped_contiguous(Ac, B, off)
    assert np.array_equal(Dc, np.concatenate([Dm[g, :mm[g]] for g in range(G)]))


def test_contiguous_swapped_weights_move_outputs():
    """Exchanging two groups' weights exchanges exactly their outputs (a
    wrong group lookup fails here)."""
    G, N, K = 3, 8, 32
    off = np.array([0, 5, 9, 16], np.int32)
    A = _rand_codes((16, K), 506, 0)
    B = _rand_codes((G, N, K), 507, 0)
    D, _ = oracle.gemm_grouped_contiguous(A, B, off)
    D2, _ = oracle.gemm_grouped_contiguous(A, B[[1, 0, 2]], off)
    ref, _ = oracle.gemm_nt(A[0:5], B[1])
    assert np.array_equal(D2[0:5], ref) and np.array_equal(D2[9:], D[9:])
