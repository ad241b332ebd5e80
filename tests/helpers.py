"""Shared helpers of the GPU parity tests: host<->device marshalling of the
oracle's bit-pattern arrays and the comparison rules.

Comparison rules (the pages fix "accumulating in fp32"; the tolerances
below are the ones the build states for it):
  * quantised codes, scales and dequantised weights: bit-exact;
  * GEMM fp32 output: |c - ref| <= 1e-4 * mag per element, where ref is the
    exact block-scaled sum and mag the same sum over absolute values; exact
    zero where mag == 0;
  * GEMM bf16 output: equal to the RNE rounding of the kernel's own fp32
    result when both are written, and within one bf16 ulp of bf16(ref)
    wherever the fp32 tolerance is below half a bf16 ulp of |ref| (elsewhere
    cancellation makes the fp32 bound the meaningful one).
"""
import numpy as np
import torch

import oracle

GEMM_RTOL = 1e-4


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_e4m3(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).cuda()


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def host_bits(t):
    """bf16 / e4m3 tensor -> numpy bit patterns (uint16 / uint8)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def host_f32(t):
    return t.detach().contiguous().cpu().numpy()


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (normal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    a = np.maximum(a, 2.0 ** -126)
    e = np.floor(np.log2(a))
    return np.exp2(e - 7)


def check_gemm(ref, mag, c_fp32=None, c_bf16=None, what=""):
    """Assert the GEMM comparison rules; returns (max err/mag, #bf16 off-by-one)."""
    ref = np.asarray(ref, np.float64)
    mag = np.asarray(mag, np.float64)
    worst = 0.0
    if c_fp32 is not None:
        c = np.asarray(c_fp32, np.float64)
        assert c.shape == ref.shape, what
        err = np.abs(c - ref)
        zero = mag == 0
        assert np.all(c[zero] == 0), f"{what}: non-zero where every product is zero"
        with np.errstate(divide="ignore", invalid="ignore"):
            rel = np.where(zero, 0.0, err / mag)
        worst = float(rel.max()) if rel.size else 0.0
        bad = rel > GEMM_RTOL
        if bad.any():
            i = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {int(bad.sum())} fp32 outputs beyond 1e-4*mag; first at {tuple(i)}: "
                                 f"got {c[tuple(i)]!r} want {ref[tuple(i)]!r} mag {mag[tuple(i)]!r}")
    off = 0
    if c_bf16 is not None:
        cb = np.asarray(c_bf16, np.uint16)
        if c_fp32 is not None:
            own = oracle.f32_to_bf16(np.asarray(c_fp32, np.float32))
            assert np.array_equal(cb, own), f"{what}: bf16 output is not the RNE rounding of the fp32 output"
        want = oracle.f32_to_bf16(ref.astype(np.float32))
        got_v = oracle.bf16_to_f32(cb).astype(np.float64)
        want_v = oracle.bf16_to_f32(want).astype(np.float64)
        ulp = bf16_ulp(ref)
        conditioned = GEMM_RTOL * mag < ulp / 2
        d = np.abs(got_v - want_v)
        assert np.all(d[conditioned] <= ulp[conditioned] * 1.0000001), f"{what}: bf16 beyond 1 ulp"
        loose = ~conditioned
        assert np.all(np.abs(got_v - ref)[loose] <= GEMM_RTOL * mag[loose] + ulp[loose]), f"{what}: bf16 band"
        off = int(np.sum(cb != want))
    return worst, off
