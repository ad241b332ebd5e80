"""GPU parity of fp8_gemm_ue8m0 -- the block-scaled product of the data-flow
page ("FP8 quantization data flow") with the optional ue8m0 scale format of
the source tour ("FP8 with per-block scales": scales rounded up to a power
of two), computed by the tensor core's block-scaled MMA -- against the
oracle's exact block-scaled sum."""
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


def _case(M, N, K, seed):
    a = syn.random_e4m3_codes((M, K), seed)
    b = syn.random_e4m3_codes((N, K), seed + 1)
    as_ = syn.random_pow2_scales((M, K // 128), seed + 2)
    bs = syn.random_pow2_scales(((N + 127) // 128, K // 128), seed + 3)
    return a, as_, b, bs


def _run(fp8, a, as_, b, bs, rows=None, what=""):
    cb, cf = fp8.fp8_gemm_ue8m0(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs), out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    ref, mag = oracle.gemm(a, as_, b, bs, rows=rows)
    cf_h, cb_h = host_f32(cf), host_bits(cb)
    if rows is not None:
        cf_h, cb_h = cf_h[rows], cb_h[rows]
    return check_gemm(ref, mag, cf_h, cb_h, what)


@pytest.mark.parametrize("shape", [(128, 256, 512), (300, 384, 1024), (129, 136, 512), (65, 8, 512),
                                   (1000, 1000, 2048), (37, 576, 7168)])
def test_random_codes_and_scales(fp8, shape):
    # one tile; ragged M and N (partial 128-row and 256-column tiles, N not a
    # multiple of 8); K of 4 slabs (fewer than the scale ring holds) up to 56
    M, N, K = shape
    _run(fp8, *_case(M, N, K, 11 + M % 13), what=f"ue8m0 {shape}")


def test_many_tiles_per_cta(fp8):
    # more tiles than SMs: each CTA moves from tile to tile, its scale writers
    # running into the next tile while the previous epilogue drains
    sms = fp8.fp8_num_sms()
    M, N, K = 16 * 128, 256 * ((3 * sms + 15) // 16), 1024
    a, as_, b, bs = _case(M, N, K, 21)
    rows = np.unique(np.r_[0:2, 127:129, 1000, 1919, M - 2:M])
    _run(fp8, a, as_, b, bs, rows=rows, what=f"many tiles {M}x{N}x{K}")


@pytest.mark.parametrize("M", [37, 2049])
def test_ragged_wkv_a(fp8, M):
    # wkv_a 7168 -> 576 with the pipeline's own ue8m0 quantisation of both operands
    lin = syn.ragged_ue8m0(M)
    aq, as_ = oracle.act_quant(lin.x, ue8m0=True)
    bq, bs = oracle.weight_quant(lin.w, ue8m0=True)
    rows = None if M < 100 else np.unique(np.r_[0:3, 127:130, 1024, M - 3:M])
    _run(fp8, aq, as_, bq, bs, rows=rows, what=f"wkv_a M={M}")


def test_prefill_w1_sampled(fp8):
    x = syn.mlp_activations(M=4096)
    aq, as_ = oracle.act_quant(x, ue8m0=True)
    w1 = syn.mlp_weight("w1", (syn.MLP_INTER, syn.MLP_DIM))
    bq, bs = oracle.weight_quant(w1, ue8m0=True)
    rng = np.random.default_rng(19)
    rows = np.unique(np.r_[0, 1, 127, 128, 4095, rng.integers(0, 4096, 9)])
    _run(fp8, aq, as_, bq, bs, rows=rows, what="w1 M=4096 ue8m0")


def test_agrees_with_fp8_gemm(fp8):
    # the same product as the per-slab promotion kernel, to the shared tolerance
    M, N, K = 512, 768, 2048
    a, as_, b, bs = _case(M, N, K, 31)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    _, c1 = fp8.fp8_gemm_ue8m0(*args, out_bf16=False, out_fp32=True)
    _, c2 = fp8.fp8_gemm(*args, out_bf16=False, out_fp32=True)
    fp8.fp8_device_status()
    ref, mag = oracle.gemm(a, as_, b, bs)
    check_gemm(ref, mag, host_f32(c1), None, "block-scaled MMA")
    check_gemm(ref, mag, host_f32(c2), None, "per-slab promotion")


@pytest.mark.parametrize("shape", [(300, 392, 512), (4100, 4736, 512)])
def test_bf16_only_output_tile_store(fp8, shape):
    # bf16-only outputs leave through TMA tile stores: bit-identical to the
    # direct stores of a call that also asks for fp32; rows past M untouched
    M, N, K = shape
    a, as_, b, bs = _case(M, N, K, 41 + M % 7)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    pad = 8
    sentinel = 0x7FBF
    buf = torch.full((M + pad, N), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fp8.fp8_gemm_ue8m0(*args, out_bf16=True, c_bf16=buf[:M])
    cb, cf = fp8.fp8_gemm_ue8m0(*args, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    got = host_bits(buf)
    assert np.all(got[M:] == sentinel), "rows past M were written"
    assert np.array_equal(got[:M], host_bits(cb)), f"{shape}: TMA-stored bf16 differs from direct stores"
    rows = np.unique(np.r_[0, 1, 31, 32, 127, 128, M // 2, M - 33, M - 1])
    ref, mag = oracle.gemm(a, as_, b, bs, rows=rows)
    check_gemm(ref, mag, host_f32(cf)[rows], got[:M][rows], f"{shape} bf16-only")


def test_repeat_calls_are_deterministic(fp8):
    a, as_, b, bs = _case(700, 1280, 1536, 51)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    outs = [host_f32(fp8.fp8_gemm_ue8m0(*args, out_bf16=False, out_fp32=True)[1]) for _ in range(3)]
    fp8.fp8_device_status()
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_scale_that_is_not_a_power_of_two_is_reported(fp8):
    a, as_, b, bs = _case(128, 256, 512, 61)
    as_[5, 2] = np.float32(1.5)   # a mantissa: not an E8M0 value
    fp8.fp8_gemm_ue8m0(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    with pytest.raises(fp8.Fp8Error) as ei:
        fp8.fp8_device_status()
    assert ei.value.status == 1   # FP8_ERR_INVALID_ARG
    fp8.fp8_device_status()       # reading cleared it


def test_k_not_a_multiple_of_512_is_rejected(fp8):
    a, as_, b, bs = _case(64, 256, 384, 71)
    with pytest.raises(fp8.Fp8Error):
        fp8.fp8_gemm_ue8m0(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))


@pytest.mark.parametrize("shape", [(2300, 2200, 1024), (4096, 2304, 512), (2049, 5120, 512)])
def test_cta_pairs_ragged(fp8, shape):
    # enough 256 x 256 tiles for the CTA-pair kernel: ragged M (the second CTA
    # of the last pair holding some or none of the rows), ragged N, repeat
    # calls bit-identical
    M, N, K = shape
    a, as_, b, bs = _case(M, N, K, 91 + M % 11)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs))
    cb, cf = fp8.fp8_gemm_ue8m0(*args, out_bf16=True, out_fp32=True)
    cf2 = fp8.fp8_gemm_ue8m0(*args, out_bf16=False, out_fp32=True)[1]
    fp8.fp8_device_status()
    assert np.array_equal(host_f32(cf), host_f32(cf2)), f"{shape}: repeat call differs"
    rows = np.unique(np.r_[0, 1, 127, 128, 129, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1])
    ref, mag = oracle.gemm(a, as_, b, bs, rows=rows)
    check_gemm(ref, mag, host_f32(cf)[rows], host_bits(cb)[rows], f"pairs {shape}")
