"""Pins of the oracle's number formats against independent implementations.

The e4m3 codec and the bf16 rounding are the base of every bit-exact
comparison.  They are pinned against torch's own float8_e4m3fn / bfloat16
conversions (a library routine written independently of the oracle) at every
rounding decision point, and against the format's definition where torch
behaves differently (torch maps magnitudes above 464 to NaN; the method
saturates).
"""
import math

import numpy as np
import pytest
import torch


def torch_e4m3_bits(v32):
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_match_library(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(codes[nan]) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], lib[~nan])
    # landmarks of the format: max finite 448, min subnormal 2^-9, min normal 2^-6
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert math.copysign(1.0, ours[0x80]) == -1.0 and ours[0x80] == 0.0


def _decision_points(orc):
    vals = orc.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448, increasing
    assert np.all(np.diff(vals) > 0)
    pts = [vals]
    mids = (vals[:-1] + vals[1:]) / 2.0                      # exact in fp32
    m32 = mids.astype(np.float32)
    assert np.array_equal(m32.astype(np.float64), mids)
    pts += [mids, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))]
    pts += [np.nextafter(vals.astype(np.float32), np.float32(np.inf)),
            np.nextafter(vals.astype(np.float32), np.float32(0))]
    p = np.concatenate([np.asarray(x, dtype=np.float32) for x in pts])
    p = p[(p >= 0) & (p <= 448)]
    return np.concatenate([p, -p])


def test_encode_at_every_decision_point_matches_library(orc):
    v = _decision_points(orc)
    assert np.array_equal(orc.e4m3_encode(v), torch_e4m3_bits(v))


def test_encode_random_sample_matches_library(orc):
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-14, np.log2(448.0), size=2_000_000)).astype(np.float32)
    sign = np.where(rng.random(mag.size) < 0.5, -1, 1).astype(np.float32)
    v = np.minimum(mag, np.float32(448)) * sign
    assert np.array_equal(orc.e4m3_encode(v), torch_e4m3_bits(v))


def test_encode_ties_go_to_even_mantissa(orc):
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even -> 0x38;
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A): even -> 0x3A;
    # 2^-10 halfway between 0 and the smallest subnormal 2^-9: even -> 0x00.
    v = np.array([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, -1.0625], dtype=np.float32)
    assert list(orc.e4m3_encode(v)) == [0x38, 0x3A, 0x00, 0x02, 0xB8]


def test_encode_saturates_beyond_max(orc):
    v = np.array([448.0, 460.0, 464.0, 465.0, 1e6, 3e38, np.inf,
                  -465.0, -np.inf], dtype=np.float32)
    assert list(orc.e4m3_encode(v)) == [0x7E] * 7 + [0xFE] * 2


def test_encode_keeps_sign_of_zero(orc):
    v = np.array([0.0, -0.0, 2.0 ** -12, -(2.0 ** -12)], dtype=np.float32)
    assert list(orc.e4m3_encode(v)) == [0x00, 0x80, 0x00, 0x80]


def test_f32_to_bf16_matches_library(orc):
    rng = np.random.default_rng(3)
    u = rng.integers(0, 2 ** 32, size=1_000_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # exact ties (low half 0x8000) with both parities of the kept bit
    ties = ((rng.integers(0, 2 ** 16, size=20000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties)]
    f = np.concatenate([f, ties, np.array([0.0, -0.0, 1.0, 3.4e38], np.float32)])
    lib = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16(f), lib)


def test_f64_to_bf16_by_construction(orc):
    L = orc.lib()
    rng = np.random.default_rng(11)
    for _ in range(2000):
        b0 = int(rng.integers(0x0080, 0x7F70))          # positive normal bf16
        lo = float(orc.bf16_to_f32(np.uint16(b0)))
        hi = float(orc.bf16_to_f32(np.uint16(b0 + 1)))
        mid = (lo + hi) / 2.0
        eps = (hi - lo) * 2.0 ** -30
        assert L.oracle_f64_to_bf16(mid + eps) == b0 + 1
        assert L.oracle_f64_to_bf16(mid - eps) == b0
        assert L.oracle_f64_to_bf16(mid) == (b0 if b0 % 2 == 0 else b0 + 1)
        assert L.oracle_f64_to_bf16(-(mid + eps)) == (b0 + 1) | 0x8000
        assert L.oracle_f64_to_bf16(lo) == b0
    # agrees with the fp32 rounding on values that fp32 holds exactly
    f = rng.standard_normal(5000).astype(np.float32)
    want = orc.f32_to_bf16(f)
    got = np.array([L.oracle_f64_to_bf16(float(x)) for x in f], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_pow2_ceil(orc):
    L = orc.lib()
    assert L.oracle_pow2_ceil(1.0) == 1.0
    assert L.oracle_pow2_ceil(0.75) == 1.0
    assert L.oracle_pow2_ceil(3.0) == 4.0
    assert L.oracle_pow2_ceil(2.0 ** -20) == 2.0 ** -20
    assert L.oracle_pow2_ceil(float(np.nextafter(np.float32(1.0), np.float32(2)))) == 2.0
    assert L.oracle_pow2_ceil(float(np.nextafter(np.float32(0.5), np.float32(0)))) == 0.5
    rng = np.random.default_rng(5)
    for s in np.exp2(rng.uniform(-30, 10, 500)).astype(np.float32):
        p = L.oracle_pow2_ceil(float(s))
        m, e = math.frexp(p)
        assert m == 0.5 and p >= s and p / 2 < s
