"""GPU parity of the dense MLP chain at its full size -- M = 4096 tokens,
7168 -> 2 x 18432 -> 7168 -- and of the GEMM at the chain's longest K range
(18432, i.e. 144 128-K slabs).

The chain is the FP8 linear of the source tour ("FP8 with per-block scales":
act_quant of the input, then the block-scaled GEMM against e4m3 weights with
128x128 scales) applied to the expert body of the behavior-traces page
("MoE trace": w2(silu(w1 x) * w3 x)), here as one dense MLP:

    x -> act_quant -> [w1 | w3] -> h1 | h3 (bf16)
      -> g = bf16(bf16(silu(h1)) * h3) -> act_quant -> w2 -> y (bf16)

Checked stage by stage: each GPU stage is compared with the oracle fed the
GPU's own output of the stage before, so differences cannot compound.  Codes
and scales bit-exact; GEMM outputs on sampled rows (first and last rows of
tiles, the last row, random rows) within 1e-4 of the exact block-scaled sum
(bf16 within 1 ulp); g within the silu rounding band.  Run with fp32 scales
on fp8_gemm, and with ue8m0 scales (weights too) on fp8_gemm_ue8m0."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import check_gemm, dev_bf16, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu

M, D, I = 4096, syn.MLP_DIM, syn.MLP_INTER


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


@pytest.fixture(scope="module")
def mlp_host():
    x = syn.mlp_activations(M=M)
    w1 = syn.mlp_weight("w1", (I, D))
    w3 = syn.mlp_weight("w3", (I, D))
    w2 = syn.mlp_weight("w2", (D, I))
    return x, w1, w3, w2


def _rows(seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.r_[0, 1, 127, 128, 129, 2047, 2048, 4095, rng.integers(0, M, 8)])


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32_scales", "ue8m0_scales"])
def test_dense_mlp_chain_stagewise(fp8, mlp_host, ue8m0):
    x, w1, w3, w2 = mlp_host
    fmt = fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32
    gemm = fp8.fp8_gemm_ue8m0 if ue8m0 else fp8.fp8_gemm
    # weights quantised by the oracle (input preparation), w1 and w3 side by side
    q1, s1 = oracle.weight_quant(w1, ue8m0=ue8m0)
    q3, s3 = oracle.weight_quant(w3, ue8m0=ue8m0)
    w13q, w13s = np.concatenate([q1, q3], 0), np.concatenate([s1, s3], 0)
    w2q, w2s = oracle.weight_quant(w2, ue8m0=ue8m0)
    del q1, q3

    # the whole chain on the GPU, bf16-only GEMM outputs (the chain's own form)
    xq, xs = fp8.fp8_act_quant(dev_bf16(x), fmt)
    h13 = gemm(xq, xs, dev_e4m3(w13q), dev_f32(w13s), out_bf16=True)[0]
    gq, gs, g = fp8.fp8_silu_mul_quant(h13, h13[:, I:], 2 * I, M, I, fmt, want_g=True)
    y = gemm(gq, gs, dev_e4m3(w2q), dev_f32(w2s), out_bf16=True)[0]
    fp8.fp8_device_status()
    xq_h, xs_h, h13_h = host_bits(xq), host_f32(xs), host_bits(h13)
    gq_h, gs_h, g_h, y_h = host_bits(gq), host_f32(gs), host_bits(g), host_bits(y)
    what = "ue8m0" if ue8m0 else "fp32"

    # 1. act_quant of x: every code and scale
    oq, os_ = oracle.act_quant(x, ue8m0=ue8m0)
    assert np.array_equal(xs_h.view(np.uint32), os_.view(np.uint32)), f"{what}: x scales"
    assert np.array_equal(xq_h, oq), f"{what}: x codes"

    # 2. w1 | w3 on sampled rows, from the GPU's codes
    rows = _rows(3 + ue8m0)
    ref, mag = oracle.gemm(xq_h, xs_h, w13q, w13s, rows=rows)
    check_gemm(ref, mag, None, h13_h[rows], f"{what}: w1|w3 (K=7168, N=36864)")

    # 3. silu * mul on the GPU's h1, h3 (sampled rows), then act_quant of the
    #    GPU's g (every row) bit-exact
    g_ref = oracle.silu_mul(h13_h[rows, :I], h13_h[rows, I:])
    gv = oracle.bf16_to_f32(g_h[rows]).astype(np.float64)
    rv = oracle.bf16_to_f32(g_ref).astype(np.float64)
    assert np.all(np.abs(gv - rv) <= 2.0 ** -6 * np.abs(rv) + 1e-30), f"{what}: g beyond the silu band"
    assert np.mean(g_h[rows] != g_ref) < 2e-3
    oq, os_ = oracle.act_quant(g_h, ue8m0=ue8m0)
    assert np.array_equal(gs_h.view(np.uint32), os_.view(np.uint32)), f"{what}: g scales"
    assert np.array_equal(gq_h, oq), f"{what}: g codes"

    # 4. w2 (K = 18432: 144 slabs, N = 7168) on sampled rows, from the GPU's codes
    rows = _rows(5 + ue8m0)
    ref, mag = oracle.gemm(gq_h, gs_h, w2q, w2s, rows=rows)
    check_gemm(ref, mag, None, y_h[rows], f"{what}: w2 (K=18432, N=7168)")


def _random_case(Mr, N, K, seed, ue8m0):
    a = syn.random_e4m3_codes((Mr, K), seed)
    b = syn.random_e4m3_codes((N, K), seed + 1)
    scales = syn.random_pow2_scales if ue8m0 else syn.random_scales
    return a, scales((Mr, K // 128), seed + 2), b, scales(((N + 127) // 128, K // 128), seed + 3)


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp8_gemm", "fp8_gemm_ue8m0"])
@pytest.mark.parametrize("shape", [(333, 384, 18432), (4100, 7168, 18432)])
def test_gemm_k18432_ragged(fp8, shape, ue8m0):
    # K = 18432 with ragged M: few tiles (split K across CTAs with fp8_gemm,
    # one 128 x 256 tile per SM with fp8_gemm_ue8m0) and the w2 shape with
    # 4 rows past the last full 256-row tile (wide tiles / CTA pairs)
    Mr, N, K = shape
    a, a_s, b, b_s = _random_case(Mr, N, K, 90 + Mr % 7, ue8m0)
    gemm = fp8.fp8_gemm_ue8m0 if ue8m0 else fp8.fp8_gemm
    cb, cf = gemm(dev_e4m3(a), dev_f32(a_s), dev_e4m3(b), dev_f32(b_s), out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    rows = np.unique(np.r_[0, 1, 127, 128, 255, 256, Mr // 2, Mr - 5:Mr])
    rows = rows[rows < Mr]
    ref, mag = oracle.gemm(a, a_s, b, b_s, rows=rows)
    check_gemm(ref, mag, host_f32(cf)[rows], host_bits(cb)[rows], f"{shape} {'ue8m0' if ue8m0 else 'fp32'}")
