"""Pins for the CPU oracle (no GPU).

Each pin checks the oracle against something other than itself: a value the
pages fix, a closed form, an exact rational brute force, or a library routine
(numpy's and the struct module's binary16 conversions).  The pins are written
as functions of a ``gemm64(A_bits, B_bits) -> float64 array`` callable so that
``test_pins_catch_planted_mistakes`` can run them against deliberately broken
copies of the oracle (planted here, on the CPU) and show that each plausible
mistake (a transposed operand, a dropped term, a flipped sign, a swapped
index, a wrong rounding) fails at least one pin.

The operation pinned is D[i][j] = sum_k A[i][k] * B[j][k] (page
"TIRx 与高性能GEMM (上)", section "从 GEMM 公式到数据路径": D = A B^T with A M x K
and B N x K; Step 3: the CTA index over A's rows selects D's row band and the
one over B's rows selects D's column band).
"""
from __future__ import annotations

import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle

F16 = np.float16


def bits(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=F16)).view(np.uint16)


def rand_f16(rng, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return bits(rng.uniform(lo, hi, size=shape))


# ---------------------------------------------------------------------------
# An independent exact reference for tiny cases: rational arithmetic and a
# brute-force nearest-binary16 search over the sorted list of all finite
# binary16 values (ties go to the even bit pattern).
# ---------------------------------------------------------------------------

def _all_finite_f16():
    pats = np.arange(0, 0x7C00, dtype=np.uint16)  # +0 .. largest finite
    vals = [Fraction(float(v)) for v in pats.view(F16).astype(np.float64)]
    return pats, vals


_POS_PATS, _POS_VALS = _all_finite_f16()


def exact_rne_f16(q: Fraction) -> int:
    """Round a rational to binary16 by brute-force search (ties to even)."""
    import bisect

    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    max_finite = _POS_VALS[-1]
    # Beyond the largest finite value, the rounding boundary is max + half an ulp (2^4).
    if a >= max_finite + Fraction(16):
        return sign | 0x7C00
    idx = bisect.bisect_left(_POS_VALS, a)
    if idx < len(_POS_VALS) and _POS_VALS[idx] == a:
        return sign | int(_POS_PATS[idx])
    lo, hi = idx - 1, idx
    if hi >= len(_POS_VALS):
        return sign | int(_POS_PATS[lo])
    dlo, dhi = a - _POS_VALS[lo], _POS_VALS[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:
        pick = lo if int(_POS_PATS[lo]) % 2 == 0 else hi
    return sign | int(_POS_PATS[pick])


def exact_gemm(A_bits, B_bits):
    a = A_bits.view(F16).astype(np.float64)
    b = B_bits.view(F16).astype(np.float64)
    M, K = a.shape
    N = b.shape[0]
    return [[sum((Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K)), Fraction(0))
             for j in range(N)] for i in range(M)]


# ---------------------------------------------------------------------------
# Pins, each parameterised by the GEMM under test.
# ---------------------------------------------------------------------------

def pin_all_ones(gemm64):
    """A = 1, B = 1 gives D = K exactly in every element."""
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 16, 64), (17, 9, 1000), (5, 3, 2048), (2, 2, 4096)]:
        A = bits(np.ones((M, K)))
        B = bits(np.ones((N, K)))
        D = gemm64(A, B)
        assert D.shape == (M, N)
        assert np.all(D == float(K)), f"all-ones {M}x{N}x{K}"


def pin_identity(gemm64):
    """B = I_K gives D = A; A = I_K gives D = B^T (every product is exact)."""
    rng = np.random.default_rng(11)
    M, K, N = 13, 24, 9
    A = rand_f16(rng, (M, K))
    D = gemm64(A, bits(np.eye(K)))
    assert np.array_equal(D, A.view(F16).astype(np.float64)), "B = I must reproduce A"
    B = rand_f16(rng, (N, K))
    D = gemm64(bits(np.eye(K)), B)
    assert np.array_equal(D, B.view(F16).astype(np.float64).T), "A = I must give B^T"


def pin_permutation(gemm64):
    """B[j, pi(j)] = 1 gives D[i, j] = A[i, pi(j)]: pins the transpose convention,
    because A * P differs from A * P^T for a non-involutive permutation."""
    rng = np.random.default_rng(12)
    M, K = 7, 16
    pi = rng.permutation(K)
    while np.array_equal(pi[pi], np.arange(K)):  # make sure P != P^T
        pi = rng.permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), pi] = 1.0
    A = rand_f16(rng, (M, K))
    D = gemm64(A, bits(P))
    a = A.view(F16).astype(np.float64)
    assert np.array_equal(D, a[:, pi]), "permutation probe"


def pin_rank_one(gemm64):
    """A = e_p u^T and B = e_q v^T give D = (u . v) at (p, q) and 0 elsewhere."""
    M, N, K = 6, 5, 12
    p, q = 4, 1
    u = np.arange(1, K + 1, dtype=np.float64) * 0.25
    v = (np.arange(K, dtype=np.float64) - 5.0) * 0.5
    A = np.zeros((M, K))
    B = np.zeros((N, K))
    A[p] = u
    B[q] = v
    D = gemm64(bits(A), bits(B))
    expect = np.zeros((M, N))
    expect[p, q] = float(sum(Fraction(x) * Fraction(y) for x, y in zip(u, v)))
    assert np.array_equal(D, expect), "rank-one probe"


def pin_bruteforce(gemm64, round_f16):
    """Random tiny cases against exact rational sums: the binary64 result is within
    a few binary64 ulps of the exact sum, and its binary16 rounding equals the
    brute-force nearest binary16 of the exact sum."""
    rng = np.random.default_rng(13)
    for M in (1, 2, 3, 7, 16):
        for (N, K) in [(1, 1), (2, 3), (3, 16), (7, 2), (16, 7)]:
            A = rand_f16(rng, (M, K))
            B = rand_f16(rng, (N, K))
            D = gemm64(A, B)
            ex = exact_gemm(A, B)
            a = A.view(F16).astype(np.float64)
            b = B.view(F16).astype(np.float64)
            mag = np.abs(a) @ np.abs(b).T
            for i in range(M):
                for j in range(N):
                    err = abs(Fraction(float(D[i, j])) - ex[i][j])
                    assert err <= Fraction(float(mag[i, j])) * Fraction(1, 2 ** 50), (M, N, K, i, j)
            got16 = round_f16(D)
            want16 = np.array([[exact_rne_f16(ex[i][j]) for j in range(N)] for i in range(M)],
                              dtype=np.uint16)
            assert np.array_equal(got16, want16), (M, N, K)


# ---------------------------------------------------------------------------
# The oracle against its pins.
# ---------------------------------------------------------------------------

def test_all_ones():
    pin_all_ones(oracle.gemm_f64)


def test_identity():
    pin_identity(oracle.gemm_f64)


def test_permutation():
    pin_permutation(oracle.gemm_f64)


def test_rank_one():
    pin_rank_one(oracle.gemm_f64)


def test_bruteforce_tiny():
    pin_bruteforce(oracle.gemm_f64, oracle.f64_to_f16_bits)


def test_all_ones_every_config_shape_sampled():
    """All-ones at every workload shape, on sampled elements (the full products
    are too large for the host): every sampled element is exactly K."""
    rng = np.random.default_rng(14)
    for (M, N, K) in [(128, 128, 64), (2048, 2048, 2048), (3000, 5000, 1000),
                      (8192, 8192, 8192), (16384, 14336, 4096)]:
        A = np.full((M, K), 0x3C00, dtype=np.uint16)  # binary16 1.0
        B = np.full((N, K), 0x3C00, dtype=np.uint16)
        rows = rng.integers(0, M, size=64)
        cols = rng.integers(0, N, size=64)
        rows[:2] = [0, M - 1]
        cols[:2] = [N - 1, 0]
        d = oracle.gemm_f64_sampled(A, B, rows, cols)
        assert np.all(d == float(K)), (M, N, K)


def test_sampled_matches_full():
    """The sampled entry point computes the same dot products as the full one."""
    rng = np.random.default_rng(15)
    A = rand_f16(rng, (37, 53))
    B = rand_f16(rng, (29, 53))
    full = oracle.gemm_f64(A, B)
    rows = rng.integers(0, 37, size=200)
    cols = rng.integers(0, 29, size=200)
    assert np.array_equal(oracle.gemm_f64_sampled(A, B, rows, cols), full[rows, cols])


def test_sampled_rejects_bad_index():
    A = np.zeros((4, 8), dtype=np.uint16)
    B = np.zeros((3, 8), dtype=np.uint16)
    with pytest.raises(IndexError):
        oracle.gemm_f64_sampled(A, B, [4], [0])
    with pytest.raises(IndexError):
        oracle.gemm_f64_sampled(A, B, [0], [3])


def test_empty_and_degenerate_shapes():
    """K = 0 is an empty sum (all zeros); M = 0 or N = 0 give empty outputs."""
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((4, 0), dtype=np.uint16)
    assert np.array_equal(oracle.gemm_f64(A, B), np.zeros((3, 4)))
    assert oracle.gemm_f64(np.zeros((0, 5), np.uint16), np.zeros((2, 5), np.uint16)).shape == (0, 2)
    assert oracle.gemm_f64(np.zeros((2, 5), np.uint16), np.zeros((0, 5), np.uint16)).shape == (2, 0)


# ---------------------------------------------------------------------------
# binary16 conversions: exhaustive and against library routines.
# ---------------------------------------------------------------------------

ALL16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def test_decode_exhaustive_vs_numpy():
    got = oracle.f16_bits_to_f64(ALL16)
    want = ALL16.view(F16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zeros keep their sign
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_encode_round_trip_exhaustive():
    vals = ALL16.view(F16).astype(np.float64)
    got = oracle.f64_to_f16_bits(vals)
    finite_or_inf = ~np.isnan(vals)
    assert np.array_equal(got[finite_or_inf], ALL16[finite_or_inf])
    assert np.all((got[~finite_or_inf] & 0x7C00) == 0x7C00)
    assert np.all((got[~finite_or_inf] & 0x3FF) != 0)


def test_encode_midpoints_ties_to_even():
    """Every midpoint between consecutive positive binary16 values goes to the even
    pattern; a hair above goes up and a hair below goes down.  Checked against the
    IEEE definition directly and against numpy and struct."""
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)  # up to the second-largest finite
    a = lo.view(F16).astype(np.float64)
    b = (lo + 1).view(F16).astype(np.float64)
    mid = (a + b) / 2  # exact in binary64
    got = oracle.f64_to_f16_bits(mid)
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    assert np.array_equal(got, mid.astype(F16).view(np.uint16))
    up = oracle.f64_to_f16_bits(np.nextafter(mid, np.inf))
    dn = oracle.f64_to_f16_bits(np.nextafter(mid, -np.inf))
    assert np.array_equal(up, lo + 1)
    assert np.array_equal(dn, lo)
    for k in range(0, lo.size, 997):  # struct's 'e' packs with round-half-even
        assert struct.unpack("<H", struct.pack("<e", float(mid[k])))[0] == got[k]


def test_encode_random_vs_numpy():
    rng = np.random.default_rng(16)
    x = np.concatenate([
        rng.standard_normal(200000) * 10.0 ** rng.uniform(-9, 5, size=200000),
        rng.uniform(-70000, 70000, size=20000),
        rng.uniform(-2.0 ** -13, 2.0 ** -13, size=20000),
    ])
    got = oracle.f64_to_f16_bits(x)
    with np.errstate(over="ignore"):   # values past 65520 round to infinity on purpose
        want = x.astype(F16).view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_special_values():
    e = oracle.f64_to_f16_bits
    assert e([65504.0])[0] == 0x7BFF
    assert e([65519.99])[0] == 0x7BFF
    assert e([65520.0])[0] == 0x7C00  # the tie at max + half ulp rounds to even: infinity
    assert e([-65520.0])[0] == 0xFC00
    assert e([1e300])[0] == 0x7C00
    assert e([2.0 ** -24])[0] == 0x0001  # smallest subnormal
    assert e([2.0 ** -25])[0] == 0x0000  # tie between 0 and 2^-24 goes to even (0)
    assert e([2.0 ** -25 * 1.0000001])[0] == 0x0001
    assert e([3 * 2.0 ** -25])[0] == 0x0002  # tie between 1 and 2 units goes to 2
    assert e([2.0 ** -14])[0] == 0x0400  # smallest normal
    assert e([2.0 ** -14 - 2.0 ** -25])[0] == 0x0400  # tie: 0x03FF is odd, rounds up
    assert e([-0.0])[0] == 0x8000
    assert e([1.0])[0] == 0x3C00
    assert e([np.inf])[0] == 0x7C00 and e([-np.inf])[0] == 0xFC00
    assert (e([np.nan])[0] & 0x7C00) == 0x7C00


def test_tolerance_formula():
    """|D_gpu - D_ref| <= 1e-3 * sqrt(K) + 2^-10 * |D_ref|, elementwise."""
    d = np.array([0.0, 1.0, -1024.0])
    t = oracle.tolerance(d, 4096)
    assert np.allclose(t, [0.064, 0.064 + 2.0 ** -10, 0.064 + 1.0])


def test_oracle_threads_reported():
    assert oracle.num_threads() >= 1


# ---------------------------------------------------------------------------
# Planted mistakes: each broken copy must fail at least one pin.
# ---------------------------------------------------------------------------

def _np_gemm64(A, B, mutate=None):
    a = A.view(F16).astype(np.float64)
    b = B.view(F16).astype(np.float64)
    M, K = a.shape
    N = b.shape[0]
    D = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            s = 0.0
            for k in range(K):
                if mutate == "dropped_term" and k == K - 1:
                    continue
                if mutate == "index_shift":
                    s += a[i, (k + 1) % K] * b[j, k]
                elif mutate == "transposed_b":
                    # treats B as K x N (computes A * B instead of A * B^T)
                    s += a[i, k] * (b[k, j] if k < N and j < K else 0.0)
                else:
                    s += a[i, k] * b[j, k]
            D[i, j] = -s if mutate == "sign" else s
    if mutate == "swapped_output" and M == N:
        D = D.T.copy()
    return D


def _truncating_round(x):
    # rounds toward zero instead of to nearest
    x = np.asarray(x, dtype=np.float64)
    out = x.astype(F16)
    over = np.abs(out.astype(np.float64)) > np.abs(x)
    out[over] = np.nextafter(out[over], F16(0))
    return out.view(np.uint16)


@pytest.mark.parametrize("mutant", ["dropped_term", "index_shift", "transposed_b", "sign",
                                    "swapped_output", "truncating_round"])
def test_pins_catch_planted_mistakes(mutant):
    gemm = (lambda A, B: _np_gemm64(A, B, None if mutant == "truncating_round" else mutant))
    rnd = _truncating_round if mutant == "truncating_round" else oracle.f64_to_f16_bits
    pins = [lambda: pin_all_ones(gemm), lambda: pin_identity(gemm),
            lambda: pin_permutation(gemm), lambda: pin_rank_one(gemm),
            lambda: pin_bruteforce(gemm, rnd)]
    failures = 0
    for p in pins:
        try:
            p()
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures >= 1, f"no pin caught the planted mistake {mutant}"


def test_unmutated_reference_copy_passes_pins():
    """The planted-mistake harness itself is sound: the unbroken numpy copy passes."""
    gemm = lambda A, B: _np_gemm64(A, B, None)  # noqa: E731
    pin_all_ones(lambda A, B: oracle.gemm_f64(A, B))  # the big all-ones shapes via the oracle
    pin_identity(gemm)
    pin_permutation(gemm)
    pin_rank_one(gemm)
    pin_bruteforce(gemm, oracle.f64_to_f16_bits)


# ---------------------------------------------------------------------------
# bfloat16 conversions and the bfloat16 GEMM.
# ---------------------------------------------------------------------------

def _torch_bf16_bits_to_f64(bits):
    import torch
    t = torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.int16).copy())
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_decode_exhaustive_vs_torch():
    got = oracle.bf16_bits_to_f64(ALL16)
    want = _torch_bf16_bits_to_f64(ALL16)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_encode_round_trip_exhaustive():
    vals = oracle.bf16_bits_to_f64(ALL16)
    got = oracle.f64_to_bf16_bits(vals)
    ok = ~np.isnan(vals)
    assert np.array_equal(got[ok], ALL16[ok])


def test_bf16_encode_midpoints_ties_to_even():
    lo = np.arange(0, 0x7F7F, dtype=np.uint16)  # positive finite, up to the second-largest
    a = oracle.bf16_bits_to_f64(lo)
    b = oracle.bf16_bits_to_f64(lo + 1)
    mid = (a + b) / 2  # exact in binary64
    got = oracle.f64_to_bf16_bits(mid)
    even = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    assert np.array_equal(oracle.f64_to_bf16_bits(np.nextafter(mid, np.inf)), lo + 1)
    assert np.array_equal(oracle.f64_to_bf16_bits(np.nextafter(mid, -np.inf)), lo)


def test_bf16_encode_vs_torch_on_binary32_values():
    """For values that are exactly binary32, torch's float32 -> bfloat16 conversion (round to
    nearest even) is a reference with no double rounding."""
    import torch
    rng = np.random.default_rng(21)
    x32 = np.concatenate([
        (rng.standard_normal(200000) * 10.0 ** rng.uniform(-30, 30, 200000)).astype(np.float32),
        rng.integers(0, 2 ** 32, 50000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x32 = x32[np.isfinite(x32)]
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_encode_special_values():
    e = oracle.f64_to_bf16_bits
    top = float(oracle.bf16_bits_to_f64(np.array([0x7F7F], np.uint16))[0])  # largest finite
    assert e([top])[0] == 0x7F7F
    assert e([top * (1 + 2.0 ** -9)])[0] == 0x7F7F           # below the halfway point
    assert e([2.0 ** 128 * (1 - 2.0 ** -9)])[0] == 0x7F80     # the tie above the top: to even (inf)
    assert e([2.0 ** -133])[0] == 0x0001 and e([2.0 ** -134])[0] == 0x0000
    assert e([-0.0])[0] == 0x8000 and e([1.0])[0] == 0x3F80
    assert e([np.inf])[0] == 0x7F80 and e([-np.inf])[0] == 0xFF80


def _bf16_bits(x):
    import torch
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_gemm_pins():
    # all ones
    for (M, N, K) in [(3, 5, 7), (17, 9, 1000)]:
        A = np.full((M, K), 0x3F80, np.uint16)
        B = np.full((N, K), 0x3F80, np.uint16)
        assert np.all(oracle.gemm_f64_dt(A, B, "bf16") == float(K))
    # permutation probe
    rng = np.random.default_rng(22)
    K = 16
    pi = rng.permutation(K)
    P = np.zeros((K, K), np.float32)
    P[np.arange(K), pi] = 1.0
    A = _bf16_bits(rng.uniform(-1, 1, (5, K)))
    D = oracle.gemm_f64_dt(A, _bf16_bits(P), "bf16")
    assert np.array_equal(D, oracle.bf16_bits_to_f64(A)[:, pi])
    # exact rational brute force, bfloat16 inputs
    for (M, N, K) in [(2, 3, 5), (4, 4, 16)]:
        A = _bf16_bits(rng.uniform(-2, 2, (M, K)))
        B = _bf16_bits(rng.uniform(-2, 2, (N, K)))
        D = oracle.gemm_f64_dt(A, B, "bf16")
        a, b = oracle.bf16_bits_to_f64(A), oracle.bf16_bits_to_f64(B)
        for i in range(M):
            for j in range(N):
                ex = sum(Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K))
                assert abs(Fraction(float(D[i, j])) - ex) <= Fraction(1, 2 ** 45)
    # the dtype-generic entry agrees with the binary16 one on binary16 data
    A = rand_f16(rng, (9, 33))
    B = rand_f16(rng, (7, 33))
    assert np.array_equal(oracle.gemm_f64_dt(A, B, "f16"), oracle.gemm_f64(A, B))


# ---------------------------------------------------------------------------
# The fused epilogue act(x + bias[j]).
# ---------------------------------------------------------------------------

def test_epilogue_bias_lands_on_columns():
    """A = 0 gives D = bias[j] in every row: pins that bias is indexed by output column."""
    M = N = 6
    bias = bits(np.arange(N, dtype=np.float64) * 0.5 - 1.0)
    X = np.zeros((M, N))
    Y = oracle.epilogue(X, bias, "none")
    assert np.array_equal(Y, np.tile(oracle.f16_bits_to_f64(bias), (M, 1)))
    assert np.array_equal(oracle.epilogue(X, None, "none"), X)


def test_epilogue_relu_closed_form():
    x = np.array([[-3.0, -0.0, 0.0, 2.5, 1e-30, -1e-30]])
    y = oracle.epilogue(x, None, "relu")
    assert np.array_equal(y, np.array([[0.0, 0.0, 0.0, 2.5, 1e-30, 0.0]]))
    bias = bits([1.0, -1.0, 0.5, -4.0, 0.0, 0.0])
    y = oracle.epilogue(np.array([[-0.5, 0.5, 0.25, 3.0, 0.0, -1.0]]), bias, "relu")
    assert np.array_equal(y, np.array([[0.5, 0.0, 0.75, 0.0, 0.0, 0.0]]))


def test_epilogue_gelu_pins():
    """GELU(x) = x * Phi(x): against scipy's normal CDF (a library routine), the odd-part
    identity GELU(x) - GELU(-x) = x, and the limits."""
    scipy_special = pytest.importorskip("scipy.special")
    x = np.linspace(-8, 8, 4001).reshape(1, -1)
    y = oracle.epilogue(x, None, "gelu")
    want = x * scipy_special.ndtr(x)
    assert np.allclose(y, want, rtol=1e-13, atol=1e-15)
    ym = oracle.epilogue(-x, None, "gelu")
    assert np.allclose(y - ym, x, rtol=0, atol=1e-14)
    assert oracle.epilogue(np.array([[0.0]]), None, "gelu")[0, 0] == 0.0
    assert abs(oracle.epilogue(np.array([[1.0]]), None, "gelu")[0, 0] - 0.8413447460685429) < 1e-15
    big = oracle.epilogue(np.array([[40.0, -40.0]]), None, "gelu")
    assert big[0, 0] == 40.0 and big[0, 1] == 0.0


def test_epilogue_sampled_matches_full():
    rng = np.random.default_rng(23)
    X = rng.standard_normal((7, 11))
    bias = bits(rng.uniform(-1, 1, 11))
    full = oracle.epilogue(X, bias, "gelu")
    rows = rng.integers(0, 7, 50)
    cols = rng.integers(0, 11, 50)
    samp = oracle.epilogue(X[rows, cols], bias, "gelu", cols=cols)
    assert np.array_equal(samp, full[rows, cols])


@pytest.mark.parametrize("mutant", ["bias_by_row", "bias_after_act", "gelu_sign"])
def test_epilogue_pins_catch_planted_mistakes(mutant):
    """Broken copies of the epilogue (planted here, on the CPU) fail the pins above."""
    scipy_special = pytest.importorskip("scipy.special")

    def broken(X, bias, act):
        X = np.array(X, dtype=np.float64)
        b = None if bias is None else oracle.f16_bits_to_f64(bias)
        if mutant == "bias_by_row" and b is not None:
            X = X + b[: X.shape[0], None]
        elif mutant != "bias_after_act" and b is not None:
            X = X + b[None, :]
        if act == "relu":
            X = np.maximum(X, 0)
        elif act == "gelu":
            s = -1.0 if mutant == "gelu_sign" else 1.0
            X = X * scipy_special.ndtr(s * X)
        if mutant == "bias_after_act" and b is not None:
            X = X + b[None, :]
        return X

    failures = 0
    M = N = 6
    bias = bits(np.arange(N, dtype=np.float64) * 0.5 - 1.0)
    try:  # bias on columns
        assert np.array_equal(broken(np.zeros((M, N)), bias, "none"),
                              np.tile(oracle.f16_bits_to_f64(bias), (M, 1)))
    except AssertionError:
        failures += 1
    try:  # relu with bias, closed form
        b2 = bits([1.0, -1.0, 0.5, -4.0, 0.0, 0.0])
        assert np.array_equal(broken(np.array([[-0.5, 0.5, 0.25, 3.0, 0.0, -1.0]]), b2, "relu"),
                              np.array([[0.5, 0.0, 0.75, 0.0, 0.0, 0.0]]))
    except AssertionError:
        failures += 1
    try:  # gelu odd-part identity, value at 1 and the large-x limit
        x = np.linspace(-4, 4, 81).reshape(1, -1)
        assert np.allclose(broken(x, None, "gelu") - broken(-x, None, "gelu"), x, atol=1e-12)
        assert abs(broken(np.array([[1.0]]), None, "gelu")[0, 0] - 0.8413447460685429) < 1e-15
        assert broken(np.array([[40.0]]), None, "gelu")[0, 0] == 40.0
    except AssertionError:
        failures += 1
    assert failures >= 1, mutant


def test_tolerance_by_dtype():
    d = np.array([0.0, 1.0, -1024.0])
    assert np.allclose(oracle.tolerance_dt(d, 4096, "f16"), oracle.tolerance(d, 4096))
    assert np.allclose(oracle.tolerance_dt(d, 4096, "bf16"), [0.064, 0.064 + 2.0 ** -7,
                                                              0.064 + 8.0])
