"""Failure detection on the GPU without a fault: every barrier wait in the
GEMM kernels is bounded, and a wait that runs out makes the kernel record
FP8_ERR_TIMEOUT, wind down (its own copies and MMAs waited for, its tensor
memory freed) and return.  The test shortens the limit to about a
millisecond through the library's test hook, withholds one hand-off in a
one-tile, one-slab GEMM, expects fp8_device_status to report the timeout,
and then checks that the next call on the same stream is exact."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import check_gemm, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu

FP8_ERR_TIMEOUT = 4


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _status(fp8):
    return fp8.lib.fp8_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_withheld_handoff_times_out_and_the_stream_recovers(fp8):
    M, N, K = 16, 128, 128     # one output tile, one 128-K slab
    a = syn.random_e4m3_codes((M, K), 201)
    b = syn.random_e4m3_codes((N, K), 202)
    a_s = syn.random_scales((M, K // 128), 203)
    b_s = syn.random_scales((1, K // 128), 204)
    args = (dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s))
    torch.cuda.synchronize()
    assert _status(fp8) == 0
    assert fp8.lib.fp8_debug_set_wait_limit(2_000_000) == 0      # ~1 ms of SM clocks
    try:
        fp8.lib.fp8_debug_skip_one_arrive()
        fp8.fp8_gemm(*args, out_bf16=True, out_fp32=True)         # launches normally
        assert _status(fp8) == FP8_ERR_TIMEOUT
        assert _status(fp8) == 0                                  # read and cleared
    finally:
        torch.cuda.synchronize()
        assert fp8.lib.fp8_debug_set_wait_limit(0) == 0
    # the hook applied to one call only; the next call is exact
    cb, cf = fp8.fp8_gemm(*args, out_bf16=True, out_fp32=True)
    assert _status(fp8) == 0
    ref, mag = oracle.gemm(a, a_s, b, b_s)
    check_gemm(ref, mag, host_f32(cf), host_bits(cb), "after the timeout")


def test_fused_gate_times_out_and_the_stream_recovers(fp8):
    # the w1|w3 kernel with the gate on warps 2-3: the epilogue's wait runs
    # out, the tile never reaches the gate warps, whose own bounded wait
    # then ends on the abort; the next call equals the unfused chain
    # 128 x 256 tiles (h1 | h3) of one 128-K slab; M large enough that the
    # unfused fp8_gemm runs the same whole-tile kernel (same fp32 order)
    M, I, K = 300, 128, 128
    a = syn.random_e4m3_codes((M, K), 211)
    w13 = syn.random_e4m3_codes((2 * I, K), 212)   # one 128-row block each of w1 and w3
    a_s = syn.random_scales((M, K // 128), 213)
    w_s = syn.random_scales((2 * I // 128, K // 128), 214)
    args = (dev_e4m3(a), dev_f32(a_s), dev_e4m3(w13), dev_f32(w_s))
    torch.cuda.synchronize()
    assert _status(fp8) == 0
    assert fp8.lib.fp8_debug_set_wait_limit(2_000_000) == 0
    try:
        fp8.lib.fp8_debug_skip_one_arrive()
        fp8.fp8_gemm_swiglu(*args)
        assert _status(fp8) == FP8_ERR_TIMEOUT
        assert _status(fp8) == 0
    finally:
        torch.cuda.synchronize()
        assert fp8.lib.fp8_debug_set_wait_limit(0) == 0
    gq, gs = fp8.fp8_gemm_swiglu(*args)
    h, _ = fp8.fp8_gemm(*args, out_bf16=True)
    yq, ys, _ = fp8.fp8_silu_mul_quant(h, h[:, I:], 2 * I, M, I)
    assert _status(fp8) == 0
    assert torch.equal(gq.view(torch.uint8), yq.view(torch.uint8))
    assert torch.equal(gs.view(torch.int32), ys.view(torch.int32))
