"""Pins of the oracle's block-scaled GEMM and its grouped (per-expert) form.

The method's product (data-flow page, "FP8 quantization data flow"; source
tour, "FP8 with per-block scales") is sum over K blocks of
a_s[m,kb] * b_s[n/128,kb] * sum_k a[m,k] b[n,k].  e4m3 values and fp32 scales
are dyadic rationals, so the exact result is computable with Python
fractions on tiny inputs: that brute force pins the oracle (a transposed
operand, a wrong scale index or a dropped block fails it).  Closed forms and
the cross-path identity of the tour (dequantise-then-matmul equals
quantise-then-fp8_gemm up to activation rounding) pin it further.
"""
from fractions import Fraction

import numpy as np
import pytest

import synthetic as syn


def exact_gemm(orc, a, a_s, b, b_s):
    M, K = a.shape
    N = b.shape[0]
    KB = K // 128
    dec = [Fraction(float(v)) if np.isfinite(v) else None for v in orc.e4m3_decode(np.arange(256))]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for kb in range(KB):
                dot = Fraction(0)
                for k in range(kb * 128, (kb + 1) * 128):
                    dot += dec[a[m, k]] * dec[b[n, k]]
                tot += Fraction(float(a_s[m, kb])) * Fraction(float(b_s[n // 128, kb])) * dot
            out[m][n] = tot
    return out


def test_brute_force_exact_rational(orc):
    M, N, K = 3, 131, 256                      # 2 N-blocks (second ragged), 2 K-blocks
    a = syn.random_e4m3_codes((M, K), 1)
    b = syn.random_e4m3_codes((N, K), 2)
    a_s = syn.random_scales((M, K // 128), 3)
    b_s = syn.random_scales((2, K // 128), 4)
    ref, mag = orc.gemm(a, a_s, b, b_s)
    ex = exact_gemm(orc, a, a_s, b, b_s)
    for m in range(M):
        for n in range(N):
            assert abs(Fraction(ref[m, n]) - ex[m][n]) <= Fraction(2) ** -50 * Fraction(mag[m, n])
    # the row-subset form returns the same rows
    r2, m2 = orc.gemm(a, a_s, b, b_s, rows=[2, 0])
    assert np.array_equal(r2, ref[[2, 0]]) and np.array_equal(m2, mag[[2, 0]])


def test_mag_is_sum_of_absolute_terms(orc):
    a = syn.random_e4m3_codes((2, 128), 5)
    b = syn.random_e4m3_codes((4, 128), 6)
    a_s = np.array([[2.0], [0.5]], np.float32)
    b_s = np.array([[3.0]], np.float32)
    ref, mag = orc.gemm(a, a_s, b, b_s)
    A = orc.e4m3_decode(a); B = orc.e4m3_decode(b)
    for m in range(2):
        for n in range(4):
            assert mag[m, n] == pytest.approx(float(np.sum(np.abs(A[m] * B[n]))) * float(a_s[m, 0]) * 3.0, rel=1e-15)


def test_identity_activation_reproduces_dequantised_weight(orc):
    # a = I (code 0x38 is 1.0) with unit scales: C[m, n] = b_s[n/128, 0] * b[n, m]
    K, N = 128, 256
    a = np.zeros((K, K), np.uint8)
    np.fill_diagonal(a, 0x38)
    a_s = np.ones((K, 1), np.float32)
    b = syn.random_e4m3_codes((N, K), 7)
    b_s = syn.random_scales((2, 1), 8)
    ref, _ = orc.gemm(a, a_s, b, b_s)
    want = (orc.e4m3_decode(b) * np.repeat(b_s.astype(np.float64), 128, 0)).T
    assert np.array_equal(ref, want)


def test_zero_scale_or_zero_codes_give_exact_zero(orc):
    a = syn.random_e4m3_codes((4, 256), 9)
    b = syn.random_e4m3_codes((128, 256), 10)
    a[:, :128] = 0
    b[:, 128:] = 0x80                            # -0.0
    ref, mag = orc.gemm(a, np.ones((4, 2), np.float32), b, np.ones((1, 2), np.float32))
    assert np.all(ref == 0) and np.all(mag == 0)


def test_cross_path_identity_of_the_two_dispatch_modes(orc):
    # bf16 mode: y = x . dequant(W)^T ; fp8 mode: y = fp8_gemm(act_quant(x), W).
    # They differ only by activation rounding, bounded per element by the
    # e4m3 round-trip bound times |w|.
    rng = np.random.default_rng(12)
    M, N, K = 5, 192, 512
    x = syn.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = syn.to_bf16_bits(0.02 * rng.standard_normal((N, K)).astype(np.float32))
    wq, ws = orc.weight_quant(w)
    xq, xs = orc.act_quant(x)
    ref, _ = orc.gemm(xq, xs, wq, ws)
    wd = syn.bf16_bits_to_f32(orc.weight_dequant(wq, ws)).astype(np.float64)
    # the exact dequantised weight (before bf16 rounding)
    wexact = orc.e4m3_decode(wq) * np.repeat(np.repeat(ws.astype(np.float64), 128, 0), 128, 1)[:N, :K]
    xf = syn.bf16_bits_to_f32(x).astype(np.float64)
    bf = xf @ wexact.T
    sc = np.repeat(xs.astype(np.float64), 128, 1)
    xerr = np.maximum(2.0 ** -4 * np.abs(xf), 2.0 ** -10 * sc)
    bound = xerr @ np.abs(wexact).T
    assert np.all(np.abs(ref - bf) <= bound * (1 + 1e-9))
    # and the bf16-rounded dequant is within half a bf16 ulp (2^-8 relative)
    assert np.all(np.abs(wd - wexact) <= 2.0 ** -8 * np.abs(wexact) * (1 + 2.0 ** -20))


def test_grouped_gemm_matches_per_group_slices(orc):
    G, N, K = 4, 136, 256
    offsets = np.array([0, 5, 5, 9, 12], np.int32)   # includes an empty group
    R = int(offsets[-1])
    a = syn.random_e4m3_codes((R, K), 13)
    a_s = syn.random_scales((R, 2), 14)
    b = syn.random_e4m3_codes((G, N, K), 15)
    b_s = syn.random_scales((G, 2, 2), 16)
    ref, mag = orc.grouped_gemm(a, a_s, b, b_s, offsets)
    for g in range(G):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        r, mg = orc.gemm(a[lo:hi], a_s[lo:hi], b[g], b_s[g])
        assert np.array_equal(ref[lo:hi], r) and np.array_equal(mag[lo:hi], mg)
    # exact brute force on the rows of one group
    ex = exact_gemm(orc, a[9:12], a_s[9:12], b[3], b_s[3])
    for i in range(3):
        for n in range(N):
            assert abs(Fraction(ref[9 + i, n]) - ex[i][n]) <= Fraction(2) ** -50 * Fraction(mag[9 + i, n])
    rr, _ = orc.grouped_gemm(a, a_s, b, b_s, offsets, rows=[11, 0])
    assert np.array_equal(rr, ref[[11, 0]])


def test_gemm_output_forms(orc):
    ref = np.array([1.0, 1.0 + 2.0 ** -30, -3.0e-5, 1.00390625], np.float64)
    f32, bf = orc.gemm_outputs(ref)
    assert f32.dtype == np.float32 and list(f32[:2]) == [1.0, 1.0]
    # 1.00390625 = 1 + 2^-8 is a bf16 tie between 1.0 and 1.0078125 -> even (1.0)
    assert bf[3] == 0x3F80
