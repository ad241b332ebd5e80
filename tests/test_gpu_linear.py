"""GPU parity of fp8_linear, the model's FP8 linear in one call (source
tour, "FP8 with per-block scales": act_quant of the activations, then
fp8_gemm).  For decode batches of up to 16 tokens the quantisation runs
inside the decode GEMM kernel; larger batches stage act_quant's codes in the
workspace.  Either way the result must equal act_quant followed by fp8_gemm
bit for bit and match the oracle's exact block-scaled product."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import check_gemm, dev_bf16, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _compare(fp8, x_bits, w_bits, ue8m0, what, expect_fused=None):
    M, K = x_bits.shape
    N = w_bits.shape[0]
    fmt = fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32
    if expect_fused is not None:
        assert (fp8.lib.fp8_linear_workspace_size(M, N, K) == 0) == expect_fused
    wq, ws = oracle.weight_quant(w_bits)
    x = dev_bf16(x_bits)
    w, w_s = dev_e4m3(wq), dev_f32(ws)
    lb, lf = fp8.fp8_linear(x, w, w_s, fmt, out_bf16=True, out_fp32=True)
    xq, xs = fp8.fp8_act_quant(x, fmt)
    gb, gf = fp8.fp8_gemm(xq, xs, w, w_s, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    assert np.array_equal(host_f32(lf).view(np.uint32), host_f32(gf).view(np.uint32)), f"{what}: fp32 differs"
    assert np.array_equal(host_bits(lb), host_bits(gb)), f"{what}: bf16 differs"
    aq, as_ = oracle.act_quant(x_bits, ue8m0=ue8m0)
    ref, mag = oracle.gemm(aq, as_, wq, ws)
    check_gemm(ref, mag, host_f32(lf), host_bits(lb), what)


@pytest.mark.parametrize("M", [1, 5, 16, 17, 32, 33, 48, 64])
def test_decode_linears(fp8, M):
    # every decode layer on the decode kernel: 16-token tiles with the
    # quantisation fused, 32- and 64-token tiles after act_quant; clusters
    # of up to 16 CTAs splitting K
    for lin in syn.decode_linears(M):
        _compare(fp8, lin.x, lin.w, False, f"{lin.name} M={M}", expect_fused=M <= 16)


def test_staged_above_64_tokens(fp8):
    # M = 65: act_quant into the workspace, then fp8_gemm
    for lin in syn.decode_linears(65, layers=["wq_a", "wo"]):
        _compare(fp8, lin.x, lin.w, False, f"{lin.name} M=65", expect_fused=False)


@pytest.mark.parametrize("shape", [(16, 128, 2048), (40, 128, 2048), (64, 40960, 256), (1, 640, 16384)])
def test_decode_cluster_and_wave_shapes(fp8, shape):
    # one tile split 16 ways (the largest cluster); 320 tiles, more than the
    # CTAs that fit at once (whole tiles in waves); a long K range at M = 1
    M, N, K = shape
    rng = np.random.default_rng(N + M)
    x = syn.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = syn.to_bf16_bits(0.02 * rng.standard_normal((N, K)).astype(np.float32))
    _compare(fp8, x, w, False, f"{M}x{N}x{K}", expect_fused=M <= 16)


@pytest.mark.parametrize("M", [23, 61])
def test_ue8m0_ragged_wider_batches(fp8, M):
    lin = syn.ragged_ue8m0(M)
    _compare(fp8, lin.x, lin.w, True, f"wkv_a M={M} ue8m0", expect_fused=False)


def test_fused_ue8m0_ragged_n(fp8):
    lin = syn.ragged_ue8m0(16)
    _compare(fp8, lin.x, lin.w, True, "wkv_a M=16 ue8m0", expect_fused=True)


@pytest.mark.parametrize("K", [1024, 7168])
def test_fused_short_k_ranges(fp8, K):
    rng = np.random.default_rng(K)
    x = syn.to_bf16_bits(rng.standard_normal((9, K)).astype(np.float32))
    w = syn.to_bf16_bits(0.02 * rng.standard_normal((1280, K)).astype(np.float32))
    _compare(fp8, x, w, False, f"9x1280x{K}", expect_fused=True)


@pytest.mark.parametrize("M", [37, 2049])
def test_ragged_ue8m0(fp8, M):
    # staged: M = 37 on the decode kernel (64-token tile), M = 2049 on the dense one
    lin = syn.ragged_ue8m0(M)
    _compare(fp8, lin.x, lin.w, True, f"wkv_a M={M} ue8m0", expect_fused=False)


def test_staged_mid_batch(fp8):
    rng = np.random.default_rng(5)
    x = syn.to_bf16_bits(rng.standard_normal((300, 1024)).astype(np.float32))
    w = syn.to_bf16_bits(0.02 * rng.standard_normal((384, 1024)).astype(np.float32))
    _compare(fp8, x, w, False, "300x384x1024", expect_fused=False)


def test_fused_special_blocks(fp8):
    # zero block, constant block and an outlier in the 16-token tile
    rng = np.random.default_rng(6)
    x = rng.standard_normal((16, 2048)).astype(np.float32)
    x[0, :128] = 0.0
    x[3, 128:256] = -2.5
    x[15, 1900] = 3e4
    w = 0.02 * rng.standard_normal((640, 2048)).astype(np.float32)
    _compare(fp8, syn.to_bf16_bits(x), syn.to_bf16_bits(w), False, "special blocks", expect_fused=True)


def test_staged_workspace_keeps_counters_clear(fp8):
    # one workspace, staged calls in a row (M = 65): both GEMMs split tiles
    # through the workspace counters, which the staged codes must not touch
    M = 65
    lins = syn.decode_linears(M, layers=["wq_a", "wq_b"])
    need = max(int(fp8.lib.fp8_linear_workspace_size(M, l.w.shape[0], l.w.shape[1])) for l in lins)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = []
    for lin in lins:
        wq, wsc = oracle.weight_quant(lin.w)
        x, w, w_s = dev_bf16(lin.x), dev_e4m3(wq), dev_f32(wsc)
        outs.append((lin, wq, wsc, fp8.fp8_linear(x, w, w_s, out_bf16=True, out_fp32=True, workspace=ws)))
    fp8.fp8_device_status()
    assert int(ws[:16384].abs().sum()) == 0, "split-tile counters left non-zero"
    for lin, wq, wsc, (lb, lf) in outs:
        aq, as_ = oracle.act_quant(lin.x)
        ref, mag = oracle.gemm(aq, as_, wq, wsc)
        check_gemm(ref, mag, host_f32(lf), host_bits(lb), f"{lin.name} M={M} shared workspace")
