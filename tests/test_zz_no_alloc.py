"""fp8_gemm_noalloc: the GEMM for callers that cannot give the library a
workspace (no cudaMalloc allowed on their path, a fixed memory budget, or an
allocator that hands out no scratch).  Its split-tile scratch is a fixed
8 MiB array inside the library.  It runs the same plan and the same
fixed-order reduction as fp8_gemm, so its outputs must equal fp8_gemm's with
a caller workspace bit for bit; two calls in a row on the same split shape
with different data (the second reusing the partial tiles the first left in
the shared array) must both be exact.

Called through the C ABI with ctypes.  Kept in its own file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import check_gemm, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    f = m.lib.fp8_gemm_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    return m


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _noalloc(fp8, a, a_s, b, b_s, M, N, K):
    cb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    cf = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = fp8.lib.fp8_gemm_noalloc(_p(a), _p(a_s), _p(b), _p(b_s), _p(cb), _p(cf), M, N, K,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, cb, cf


def _case(M, N, K, seed):
    aq = syn.random_e4m3_codes((M, K), seed)
    bq = syn.random_e4m3_codes((N, K), seed + 1)
    as_ = syn.random_scales((M, K // 128), seed + 2)
    bs = syn.random_scales(((N + 127) // 128, K // 128), seed + 3)
    return aq, as_, bq, bs


def test_two_calls_in_a_row_match_the_workspace_entry_point(fp8):
    # shapes with few output tiles: K is split across CTAs with partial tiles
    # in the scratch.  Each shape runs twice in a row with different data, so
    # the second call overwrites the partials the first one left behind.
    cases = [(300, 384, 1024, 40), (300, 384, 1024, 60), (129, 136, 256, 50), (129, 136, 256, 70)]
    results = []
    for M, N, K, seed in cases:
        name = f"{M}x{N}x{K} seed {seed}"
        aq, as_, bq, bs = _case(M, N, K, seed)
        assert 0 < fp8.fp8_gemm_workspace_size(M, N, K) <= SCRATCH_BYTES
        args = (dev_e4m3(aq), dev_f32(as_), dev_e4m3(bq), dev_f32(bs))
        st, cb, cf = _noalloc(fp8, *args, M, N, K)
        assert st == 0, fp8.lib.fp8_status_string(st)
        results.append((name, aq, as_, bq, bs, args, cb, cf))
    fp8.fp8_device_status()
    for name, aq, as_, bq, bs, args, cb, cf in results:
        ref, mag = oracle.gemm(aq, as_, bq, bs)
        check_gemm(ref, mag, host_f32(cf), host_bits(cb), f"noalloc {name}")
        wb, wf = fp8.fp8_gemm(*args, out_bf16=True, out_fp32=True)
        fp8.fp8_device_status()
        assert np.array_equal(host_f32(cf).view(np.uint32), host_f32(wf).view(np.uint32)), \
            f"{name}: fp32 output differs from fp8_gemm's"
        assert np.array_equal(host_bits(cb), host_bits(wb)), f"{name}: bf16 output differs from fp8_gemm's"


def test_rejected_call_enqueues_nothing(fp8):
    # a misaligned operand is rejected before the shared array is touched
    M, N, K = 300, 384, 1024
    aq, as_, bq, bs = _case(M, N, K, 80)
    a, s_a, b, s_b = dev_e4m3(aq), dev_f32(as_), dev_e4m3(bq), dev_f32(bs)
    raw = torch.empty(M * K + 16, dtype=torch.uint8, device="cuda")
    a_mis = raw[1:1 + M * K].view(M, K)
    st, _, _ = _noalloc(fp8, a_mis, s_a, b, s_b, M, N, K)
    assert st == 1   # FP8_ERR_INVALID_ARG
    # the next call still finds clean counters and is exact
    st, cb, cf = _noalloc(fp8, a, s_a, b, s_b, M, N, K)
    assert st == 0
    fp8.fp8_device_status()
    wb, wf = fp8.fp8_gemm(a, s_a, b, s_b, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    assert np.array_equal(host_f32(cf).view(np.uint32), host_f32(wf).view(np.uint32))


def test_shapes_needing_more_scratch_are_rejected(fp8):
    # 64 output tiles of 128 x 128 over K = 8192: stream-K partials of
    # ~20 MB on 152 SMs
    M, N, K = 1024, 1024, 8192
    if fp8.fp8_gemm_workspace_size(M, N, K) <= SCRATCH_BYTES:
        pytest.skip("this device's schedule fits the fixed scratch")
    a = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    s = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    b = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    bs = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    st, _, _ = _noalloc(fp8, a, s, b, bs, M, N, K)
    assert st == 5   # FP8_ERR_WORKSPACE: nothing launched
