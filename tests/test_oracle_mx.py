"""Pins for the block-scaled FP8 oracle (oracle/mx_ref.c), none of which re-types its formula.

* the FP8 decoders against torch's float8_e4m3fn / float8_e5m2 conversions (a library routine),
  exhaustively, and against values fixed by the formats' definitions;
* E5M2 against the binary16 decoder (an E5M2 code is the high byte of a binary16 pattern);
* the E8M0 decoder against its closed form 2^(e - 127);
* the GEMM with unit scales against the (separately pinned) binary16 GEMM;
* closed forms for all-ones operands under arbitrary scales, and for a single live block;
* exact rational brute force on tiny inputs;
* planted mistakes in a numpy copy of the oracle, each of which some pin must catch.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _torch_fp8_to_f64(codes: np.ndarray, fmt: str) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return t.view(dt).to(torch.float64).numpy()


def _finite_codes(fmt: str) -> np.ndarray:
    c = np.arange(256, dtype=np.uint8)
    v = _torch_fp8_to_f64(c, fmt)
    return c[np.isfinite(v)]


def _rand_codes(rng, shape, fmt="e4m3"):
    ok = _finite_codes(fmt)
    return ok[rng.integers(0, ok.size, size=shape)].astype(np.uint8)


# ---- decoders -----------------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_decode_exhaustive_vs_torch(fmt):
    c = np.arange(256, dtype=np.uint8)
    ours = oracle.fp8_bits_to_f64(c, fmt)
    ref = _torch_fp8_to_f64(c, fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_fp8_values_fixed_by_the_formats():
    e4 = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
          0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in e4.items():
        assert oracle.fp8_bits_to_f64(np.array([code], np.uint8), "e4m3")[0] == val, hex(code)
    assert math.isnan(oracle.fp8_bits_to_f64(np.array([0x7F], np.uint8), "e4m3")[0])
    assert math.isnan(oracle.fp8_bits_to_f64(np.array([0xFF], np.uint8), "e4m3")[0])
    assert np.signbit(oracle.fp8_bits_to_f64(np.array([0x80], np.uint8), "e4m3")[0])
    # E4M3 has no infinities: every exponent-15 code but the NaN is a finite number
    assert np.all(np.isfinite(oracle.fp8_bits_to_f64(np.arange(0x78, 0x7F, dtype=np.uint8),
                                                     "e4m3")))
    e5 = {0x01: 2.0 ** -16, 0x04: 2.0 ** -14, 0x3C: 1.0, 0x7B: 57344.0, 0x7C: math.inf,
          0xFC: -math.inf}
    for code, val in e5.items():
        assert oracle.fp8_bits_to_f64(np.array([code], np.uint8), "e5m2")[0] == val, hex(code)
    for code in (0x7D, 0x7E, 0x7F, 0xFD):
        assert math.isnan(oracle.fp8_bits_to_f64(np.array([code], np.uint8), "e5m2")[0])


def test_e5m2_is_the_high_byte_of_binary16():
    c = np.arange(256, dtype=np.uint8)
    e5 = oracle.fp8_bits_to_f64(c, "e5m2")
    h = oracle.f16_bits_to_f64(c.astype(np.uint16) << 8)
    nan = np.isnan(h)
    assert np.array_equal(np.isnan(e5), nan)
    assert np.array_equal(e5[~nan], h[~nan])


def test_e8m0_closed_form():
    c = np.arange(256, dtype=np.uint8)
    s = oracle.e8m0_to_f64(c)
    for e in range(255):
        assert s[e] == 2.0 ** (e - 127), e
    assert math.isnan(s[255])
    assert s[127] == 1.0 and s[0] == 2.0 ** -127 and s[254] == 2.0 ** 127


# ---- the GEMM: pins written as functions of (gemm, decode) so the mutants can run them ---------

def pin_unit_scales_reduce_to_f16_gemm(gemm):
    """All scales 2^0: D equals the binary16 GEMM of the decoded elements (every E4M3 and E5M2
    value is a binary16 value), and Dabs the binary16 GEMM of their magnitudes."""
    rng = np.random.default_rng(1)
    M, N, K = 9, 7, 96
    fails = 0
    for fa, fb in (("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e5m2", "e5m2")):
        A = _rand_codes(rng, (M, K), fa)
        B = _rand_codes(rng, (N, K), fb)
        if fa == "e5m2":   # keep E5M2 magnitudes where binary16 sums stay finite
            A = np.where(np.abs(_torch_fp8_to_f64(A, fa)) <= 16.0, A, 0x3C).astype(np.uint8)
        if fb == "e5m2":
            B = np.where(np.abs(_torch_fp8_to_f64(B, fb)) <= 16.0, B, 0x3C).astype(np.uint8)
        SA = np.full((M, K // 32), 127, np.uint8)
        SB = np.full((N, K // 32), 127, np.uint8)
        D, Dabs = gemm(A, B, SA, SB, fa, fb)
        a16 = _torch_fp8_to_f64(A, fa).astype(np.float16)
        b16 = _torch_fp8_to_f64(B, fb).astype(np.float16)
        ref = oracle.gemm_f64(a16, b16)
        ref_abs = oracle.gemm_f64(np.abs(a16), np.abs(b16))
        fails += int(not np.array_equal(D, ref)) + int(not np.array_equal(Dabs, ref_abs))
    return fails


def pin_all_ones_closed_form(gemm):
    """A = B = 1.0 everywhere: D[i][j] = 32 * sum_b 2^(SA[i][b] + SB[j][b] - 254), exactly
    (scales within +-7 of 127 keep every partial sum exact in binary64)."""
    rng = np.random.default_rng(2)
    M, N, K = 5, 6, 160
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    SA = rng.integers(120, 135, size=(M, K // 32)).astype(np.uint8)
    SB = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    D, Dabs = gemm(A, B, SA, SB, "e4m3", "e4m3")
    fails = 0
    for i in range(M):
        for j in range(N):
            exact = sum(32 * Fraction(2) ** (int(SA[i, b]) + int(SB[j, b]) - 254)
                        for b in range(K // 32))
            fails += int(Fraction(D[i, j]) != exact) + int(Fraction(Dabs[i, j]) != exact)
    return fails


def pin_single_live_block(gemm):
    """Only block b of A is nonzero: D = 2^(SA[i][b] + SB[j][b] - 254) * sum over that block."""
    rng = np.random.default_rng(3)
    M, N, K = 4, 3, 128
    fails = 0
    for b in range(K // 32):
        A = np.zeros((M, K), np.uint8)
        A[:, 32 * b:32 * b + 32] = _rand_codes(rng, (M, 32))
        B = _rand_codes(rng, (N, K))
        SA = rng.integers(121, 134, size=(M, K // 32)).astype(np.uint8)
        SB = rng.integers(121, 134, size=(N, K // 32)).astype(np.uint8)
        D, _ = gemm(A, B, SA, SB, "e4m3", "e4m3")
        a = _torch_fp8_to_f64(A, "e4m3")
        bb = _torch_fp8_to_f64(B, "e4m3")
        for i in range(M):
            for j in range(N):
                blk = sum(Fraction(a[i, k]) * Fraction(bb[j, k])
                          for k in range(32 * b, 32 * b + 32))
                exact = Fraction(2) ** (int(SA[i, b]) + int(SB[j, b]) - 254) * blk
                fails += int(Fraction(D[i, j]) != exact)
    return fails


def pin_bruteforce(gemm):
    """Tiny random problems against an exact rational sum: |D - exact| <= K 2^-53 Dabs_exact and
    Dabs within the same bound."""
    rng = np.random.default_rng(4)
    fails = 0
    for (M, N, K) in ((1, 1, 32), (2, 3, 64), (3, 2, 96), (4, 4, 32)):
        for fa, fb in (("e4m3", "e4m3"), ("e4m3", "e5m2")):
            A = _rand_codes(rng, (M, K), fa)
            B = _rand_codes(rng, (N, K), fb)
            SA = rng.integers(118, 137, size=(M, K // 32)).astype(np.uint8)
            SB = rng.integers(118, 137, size=(N, K // 32)).astype(np.uint8)
            D, Dabs = gemm(A, B, SA, SB, fa, fb)
            a = _torch_fp8_to_f64(A, fa)
            b = _torch_fp8_to_f64(B, fb)
            for i in range(M):
                for j in range(N):
                    terms = [Fraction(a[i, k]) * Fraction(2) ** (int(SA[i, k // 32]) - 127)
                             * Fraction(b[j, k]) * Fraction(2) ** (int(SB[j, k // 32]) - 127)
                             for k in range(K)]
                    exact = sum(terms)
                    exact_abs = sum(abs(t) for t in terms)
                    bound = K * Fraction(2) ** -53 * exact_abs
                    fails += int(abs(Fraction(D[i, j]) - exact) > bound)
                    fails += int(abs(Fraction(Dabs[i, j]) - exact_abs) > bound)
    return fails


PINS = [pin_unit_scales_reduce_to_f16_gemm, pin_all_ones_closed_form, pin_single_live_block,
        pin_bruteforce]


def _oracle_gemm(A, B, SA, SB, fa, fb):
    return oracle.gemm_mx_f64(A, B, SA, SB, fa, fb)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(_oracle_gemm) == 0


def test_sampled_matches_full():
    rng = np.random.default_rng(5)
    M, N, K = 37, 29, 224
    A, B = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K), "e5m2")
    SA = rng.integers(120, 135, size=(M, K // 32)).astype(np.uint8)
    SB = rng.integers(120, 135, size=(N, K // 32)).astype(np.uint8)
    D, Dabs = oracle.gemm_mx_f64(A, B, SA, SB, "e4m3", "e5m2")
    r = rng.integers(0, M, 200)
    c = rng.integers(0, N, 200)
    s, sa = oracle.gemm_mx_f64_sampled(A, B, SA, SB, r, c, "e4m3", "e5m2")
    assert np.array_equal(s, D[r, c]) and np.array_equal(sa, Dabs[r, c])


def test_shape_checks():
    A = np.zeros((4, 48), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_mx_f64(A, A, np.zeros((4, 1), np.uint8), np.zeros((4, 1), np.uint8))
    A = np.zeros((4, 64), np.uint8)
    with pytest.raises(ValueError):
        oracle.gemm_mx_f64(A, A, np.zeros((4, 3), np.uint8), np.zeros((4, 2), np.uint8))
    with pytest.raises(IndexError):
        oracle.gemm_mx_f64_sampled(A, A, np.zeros((4, 2), np.uint8), np.zeros((4, 2), np.uint8),
                                   [4], [0])


def test_nan_scale_and_nan_element_propagate():
    A = np.full((2, 32), 0x38, np.uint8)
    SA = np.full((2, 1), 127, np.uint8)
    SB = SA.copy()
    SB[1, 0] = 255
    D, _ = oracle.gemm_mx_f64(A, A, SA, SB)
    assert np.isfinite(D[:, 0]).all() and np.isnan(D[:, 1]).all()
    A2 = A.copy()
    A2[0, 5] = 0x7F
    D, _ = oracle.gemm_mx_f64(A2, A, SA, SA)
    assert np.isnan(D[0]).all() and np.isfinite(D[1]).all()


def test_tolerance_mx_formula():
    d = np.array([0.0, 1.0, -1024.0])
    da = np.array([0.0, 2.0, 4096.0])
    t = oracle.tolerance_mx(d, da, 4096, "f16")
    assert np.allclose(t, np.abs(d) * 2.0 ** -10 + 4 * 129 * 2.0 ** -24 * da, rtol=0, atol=0)
    t = oracle.tolerance_mx(d, da, 4096, "bf16")
    assert np.allclose(t, np.abs(d) * 2.0 ** -7 + 4 * 129 * 2.0 ** -24 * da, rtol=0, atol=0)


# ---- planted mistakes -----------------------------------------------------------------------------

def _np_decode_fp8(c, fmt, mutant=None):
    c = np.asarray(c, dtype=np.int64)
    s = np.where((c >> 7) & 1, -1.0, 1.0)
    if fmt == "e4m3":
        e, f = (c >> 3) & 15, c & 7
        bias = 8 if mutant == "e4m3_bias8" else 7
        normal = (1 + f / 8.0) * np.exp2(e - bias)
        sub = (f / 8.0) * np.exp2(1 - bias)
        if mutant == "no_subnormals":
            sub = normal
        v = np.where(e == 0, sub, normal)
        v = np.where((e == 15) & (f == 7), np.nan, v)
    else:
        e, f = (c >> 2) & 31, c & 3
        v = np.where(e == 0, (f / 4.0) * 2.0 ** -14, (1 + f / 4.0) * np.exp2(e - 15))
        v = np.where(e == 31, np.where(f == 0, np.inf, np.nan), v)
    return s * v


def _np_gemm_mx(mutant=None):
    def gemm(A, B, SA, SB, fa, fb):
        K = A.shape[1]
        blk = 16 if mutant == "block16" else 32
        ka = np.arange(K) // blk
        ka = np.minimum(ka, SA.shape[1] - 1)
        sa = np.exp2(SA.astype(np.float64)[:, ka] - 127)
        sb = np.exp2(SB.astype(np.float64)[:, ka] - (126 if mutant == "scale_bias126" else 127))
        if mutant == "drop_sb":
            sb = np.ones_like(sb)
        if mutant == "scale_by_col" and SA.shape[0] == SB.shape[0]:
            sa, sb = sb, sa
        elif mutant == "scale_by_col":
            sa = np.exp2(SA.astype(np.float64)[::-1][:, ka] - 127)
        a = _np_decode_fp8(A, fa, mutant) * sa
        b = _np_decode_fp8(B, fb, mutant) * sb
        if mutant == "dropped_last_block":
            a = a.copy()
            a[:, K - 32:] = 0.0
        D = a @ b.T
        Dabs = np.abs(a) @ np.abs(b).T
        return D, Dabs
    return gemm


MUTANTS = ["block16", "scale_bias126", "drop_sb", "scale_by_col", "e4m3_bias8",
           "no_subnormals", "dropped_last_block"]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistakes(mutant):
    g = _np_gemm_mx(mutant)
    assert sum(pin(g) for pin in PINS) >= 1, f"no pin caught {mutant}"


def test_unmutated_numpy_copy_passes_the_exact_pins():
    g = _np_gemm_mx(None)
    # numpy's matmul sums in its own order, so only the pins exact under any order apply
    assert pin_all_ones_closed_form(g) == 0
    assert pin_bruteforce(g) == 0
