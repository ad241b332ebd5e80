"""GPU parity of fp8_gemm (data-flow page, "FP8 quantization data flow";
source tour, "FP8 with per-block scales") against the oracle's exact
block-scaled sum, on the decode (operand-swapped, stream-K), ragged,
prefill (data-parallel) and tiny workloads."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import check_gemm, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _run(fp8, aq, as_, bq, bs, rows=None, what=""):
    cb, cf = fp8.fp8_gemm(dev_e4m3(aq), dev_f32(as_), dev_e4m3(bq), dev_f32(bs), out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    ref, mag = oracle.gemm(aq, as_, bq, bs, rows=rows)
    cf_h, cb_h = host_f32(cf), host_bits(cb)
    if rows is not None:
        cf_h, cb_h = cf_h[rows], cb_h[rows]
    return check_gemm(ref, mag, cf_h, cb_h, what)


def _quantised(lin, ue8m0=False):
    aq, as_ = oracle.act_quant(lin.x, ue8m0=ue8m0)
    bq, bs = oracle.weight_quant(lin.w)
    return aq, as_, bq, bs


def test_single_tile_random_codes(fp8):
    # one 128x16 swapped tile, one slab: the smallest tensor-core path
    a = syn.random_e4m3_codes((16, 128), 1)
    b = syn.random_e4m3_codes((128, 128), 2)
    _run(fp8, a, np.ones((16, 1), np.float32), b, np.ones((1, 1), np.float32), what="single tile")


def test_tiny_linear(fp8):
    _run(fp8, *_quantised(syn.tiny_linear()), what="tiny")


@pytest.mark.parametrize("M", [1, 16, 64])
def test_decode_linears(fp8, M):
    for lin in syn.decode_linears(M):
        _run(fp8, *_quantised(lin), what=f"{lin.name} M={M}")


@pytest.mark.parametrize("M", [2, 5, 17, 33, 48])
def test_decode_odd_batches(fp8, M):
    lin = syn.decode_linears(M, layers=["wq_a"])[0]
    _run(fp8, *_quantised(lin), what=f"wq_a M={M}")


@pytest.mark.parametrize("M", [37, 2049])
def test_ragged_n_ue8m0(fp8, M):
    _run(fp8, *_quantised(syn.ragged_ue8m0(M), ue8m0=True), what=f"wkv_a M={M}")


@pytest.mark.parametrize("shape", [(300, 384, 1024), (129, 136, 256), (65, 8, 128), (200, 1000, 384)])
def test_ragged_non_swapped(fp8, shape):
    M, N, K = shape
    a = syn.random_e4m3_codes((M, K), M)
    b = syn.random_e4m3_codes((N, K), N)
    as_ = syn.random_scales((M, K // 128), 3)
    bs = syn.random_scales(((N + 127) // 128, K // 128), 4)
    _run(fp8, a, as_, b, bs, what=f"ragged {shape}")


def test_data_parallel_schedule(fp8):
    # >= 4 tiles per SM: whole tiles per CTA, no workspace
    sms = fp8.fp8_num_sms()
    M, N, K = 2048, 128 * ((4 * sms + 15) // 16), 256
    assert fp8.fp8_gemm_workspace_size(M, N, K) == 0
    a = syn.random_e4m3_codes((M, K), 5)
    b = syn.random_e4m3_codes((N, K), 6)
    as_ = syn.random_scales((M, K // 128), 7)
    bs = syn.random_scales(((N + 127) // 128, K // 128), 8)
    rows = np.r_[0:3, 127:130, 1000, M - 2:M]
    _run(fp8, a, as_, b, bs, rows=rows, what="data-parallel")


@pytest.mark.parametrize("shape", [(4100, 4736, 256), (4300, 4864, 384)])
def test_wide_tile_schedule_ragged(fp8, shape):
    # enough 128x256 tiles for whole-tile scheduling, ragged in M (last tile
    # with 4 or 76 valid rows) and in N (the last tile's upper 128 columns lie
    # past N for 4736, not for 4864)
    M, N, K = shape
    a = syn.random_e4m3_codes((M, K), 31)
    b = syn.random_e4m3_codes((N, K), 32)
    as_ = syn.random_scales((M, K // 128), 33)
    bs = syn.random_scales(((N + 127) // 128, K // 128), 34)
    rows = np.unique(np.r_[0:2, 127:129, 255:257, 2047, 4095:4098, 4223:4226, M - 3:M])
    rows = rows[rows < M]
    _run(fp8, a, as_, b, bs, rows=rows, what=f"wide tiles {shape}")


def test_prefill_mlp_shapes_sampled(fp8):
    x = syn.mlp_activations(M=4096)
    aq, as_ = oracle.act_quant(x)
    rng = np.random.default_rng(9)
    rows = np.unique(np.r_[0, 1, 127, 128, 4095, rng.integers(0, 4096, 11)])
    w1 = syn.mlp_weight("w1", (syn.MLP_INTER, syn.MLP_DIM))
    bq, bs = oracle.weight_quant(w1)
    _run(fp8, aq, as_, bq, bs, rows=rows, what="w1 M=4096")


def _random_case(M, N, K, seed):
    a = syn.random_e4m3_codes((M, K), seed)
    b = syn.random_e4m3_codes((N, K), seed + 1)
    as_ = syn.random_scales((M, K // 128), seed + 2)
    bs = syn.random_scales(((N + 127) // 128, K // 128), seed + 3)
    return a, as_, b, bs


def test_workspace_too_small_is_reported(fp8):
    # few output tiles: K split across CTAs with partials in the workspace
    M, N, K = 300, 384, 1024
    need = fp8.fp8_gemm_workspace_size(M, N, K)
    assert need > 0
    a, as_, b, bs = _random_case(M, N, K, 50)
    ws = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8.Fp8Error) as ei:
        fp8.fp8_gemm(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs), workspace=ws)
    assert ei.value.status == 5


@pytest.mark.parametrize("M", [1, 16, 33, 64])
def test_decode_shapes_need_no_workspace(fp8, M):
    # cluster split-K on chip, or whole tiles when they outnumber the slots
    for N, K in syn.DECODE_LAYERS.values():
        assert fp8.fp8_gemm_workspace_size(M, N, K) == 0


@pytest.mark.parametrize("layer", ["wq_a", "wo"])
def test_cluster_split_is_deterministic(fp8, layer):
    lin = syn.decode_linears(16, layers=[layer])[0]
    args = tuple(f(v) for f, v in zip((dev_e4m3, dev_f32, dev_e4m3, dev_f32), _quantised(lin)))
    outs = [host_f32(fp8.fp8_gemm(*args, out_bf16=False, out_fp32=True)[1]) for _ in range(3)]
    fp8.fp8_device_status()
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_repeat_calls_are_deterministic_and_leave_workspace_clean(fp8):
    M, N, K = 300, 384, 1024
    a, as_, b, bs = _random_case(M, N, K, 60)
    need = fp8.fp8_gemm_workspace_size(M, N, K)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    outs = [host_f32(fp8.fp8_gemm(*args, out_bf16=False, out_fp32=True, workspace=ws)[1]) for _ in range(3)]
    fp8.fp8_device_status()
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    # counters region (first 16 KiB) returns to zero
    cnt = ws[: 16384].view(torch.int32)
    assert int(cnt.abs().sum()) == 0


def test_one_workspace_serves_shapes_in_any_order(fp8):
    # a call with few split tiles leaves partials where a later call with
    # more split tiles keeps counters: counters must live apart from partials
    shapes = [(129, 136, 256), (1024, 1152, 8192), (300, 384, 1024), (1024, 1152, 8192), (129, 136, 256)]
    ws = torch.zeros(max(fp8.fp8_gemm_workspace_size(*sh) for sh in shapes), dtype=torch.uint8, device="cuda")
    for i, (M, N, K) in enumerate(shapes):
        assert fp8.fp8_gemm_workspace_size(M, N, K) > 0
        a, as_, b, bs = _random_case(M, N, K, 70 + i)
        cb, cf = fp8.fp8_gemm(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs), out_fp32=True, workspace=ws)
        fp8.fp8_device_status()
        rows = None if M * N <= 1 << 20 else np.r_[0:3, M - 3:M]
        ref, mag = oracle.gemm(a, as_, b, bs, rows=rows)
        cf_h, cb_h = host_f32(cf), host_bits(cb)
        if rows is not None:
            cf_h, cb_h = cf_h[rows], cb_h[rows]
        check_gemm(ref, mag, cf_h, cb_h, f"{M}x{N}x{K} shared workspace")


@pytest.mark.parametrize("shape", [(300, 392, 256), (1000, 1000, 384), (2048, 4864, 256), (4100, 4736, 256)])
def test_bf16_only_output_tile_store(fp8, shape):
    # bf16-only outputs of the non-swapped layout leave through shared memory
    # and TMA stores: bit-identical to the direct stores of a call that also
    # asks for fp32, clipped at the ragged edges (rows past M stay untouched)
    M, N, K = shape
    a, as_, b, bs = _random_case(M, N, K, 80 + M % 17)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    pad = 8
    sentinel = 0x7FBF
    buf = torch.full((M + pad, N), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fp8.fp8_gemm(*args, out_bf16=True, c_bf16=buf[:M])
    cb, cf = fp8.fp8_gemm(*args, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    got = host_bits(buf)
    assert np.all(got[M:] == sentinel), "rows past M were written"
    assert np.array_equal(got[:M], host_bits(cb)), f"{shape}: TMA-stored bf16 differs from direct stores"
    rows = np.unique(np.r_[0, 1, 31, 32, 127, 128, M // 2, M - 33, M - 1])
    ref, mag = oracle.gemm(a, as_, b, bs, rows=rows)
    check_gemm(ref, mag, host_f32(cf)[rows], got[:M][rows], f"{shape} bf16-only")
