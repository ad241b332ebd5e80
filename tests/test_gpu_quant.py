"""GPU parity of the bandwidth-bound kernels against the oracle, bit-exact:
act_quant (data-flow page, "FP8 quantization data flow"; source tour, "FP8
with per-block scales"), 128x128 weight quantisation, weight_dequant
(behavior-traces page, "fp8->bf16 trace") and the fused silu*mul+act_quant
of the expert body."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import dev_bf16, dev_e4m3, dev_f32, host_bits, host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _act_case(fp8, x_bits, ue8m0):
    y, s = fp8.fp8_act_quant(dev_bf16(x_bits), fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32)
    torch.cuda.synchronize()
    yo, so = oracle.act_quant(x_bits, ue8m0=ue8m0)
    assert np.array_equal(host_f32(s).view(np.uint32), so.view(np.uint32)), "scales differ"
    got = host_bits(y)
    if not np.array_equal(got, yo):
        bad = np.argwhere(got != yo)
        raise AssertionError(f"{len(bad)} codes differ, first at {tuple(bad[0])}: {got[tuple(bad[0])]:#x} vs {yo[tuple(bad[0])]:#x}")


@pytest.mark.parametrize("ue8m0", [False, True])
def test_act_quant_tiny(fp8, ue8m0):
    _act_case(fp8, syn.tiny_linear().x, ue8m0)


@pytest.mark.parametrize("M", [1, 16, 64])
def test_act_quant_decode_shapes(fp8, M):
    for lin in syn.decode_linears(M):
        _act_case(fp8, lin.x, False)


@pytest.mark.parametrize("M", [37, 2049])
def test_act_quant_ragged_ue8m0_with_special_blocks(fp8, M):
    lin = syn.ragged_ue8m0(M)
    _act_case(fp8, lin.x, True)
    _act_case(fp8, lin.x, False)


def test_act_quant_prefill_activations(fp8):
    x = syn.mlp_activations(M=4096)
    _act_case(fp8, x, False)


def test_act_quant_wide_dynamic_range(fp8):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((300, 1024)).astype(np.float32)
    x *= np.exp2(rng.integers(-30, 30, size=(300, 8, 1))).repeat(128, 2).reshape(300, 1024)
    x[5, :128] = 0.0
    x[6, 128:256] = -0.0
    x[7, 256:384] = 2.0 ** -120          # below the floor: scale is the floor's
    _act_case(fp8, syn.to_bf16_bits(x), False)
    _act_case(fp8, syn.to_bf16_bits(x), True)


def test_act_quant_empty_is_noop(fp8):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    y, s = fp8.fp8_act_quant(x)
    assert y.shape == (0, 256) and s.shape == (0, 2)


@pytest.mark.parametrize("shape", [(256, 256), (576, 7168), (300, 384), (130, 144)])
def test_weight_quant(fp8, shape):
    w = syn.normal_bf16(np.random.default_rng(sum(shape)), shape, 0.02)
    w[:1, :16] = 0
    q, s = fp8.fp8_weight_quant(dev_bf16(w))
    qo, so = oracle.weight_quant(w)
    assert np.array_equal(host_f32(s), so)
    assert np.array_equal(host_bits(q), qo)


def test_weight_quant_ragged_special_blocks(fp8):
    lin = syn.ragged_ue8m0(37)
    q, s = fp8.fp8_weight_quant(dev_bf16(lin.w))
    qo, so = oracle.weight_quant(lin.w)
    assert np.array_equal(host_f32(s), so)
    assert np.array_equal(host_bits(q), qo)


def test_weight_dequant_full_size(fp8):
    w = syn.dequant_source()
    wq, ws = oracle.weight_quant(w)
    y = fp8.fp8_weight_dequant(dev_e4m3(wq), dev_f32(ws))
    yo = oracle.weight_dequant(wq, ws)
    assert np.array_equal(host_bits(y), yo)


@pytest.mark.parametrize("shape", [(300, 272), (128, 16), (1, 4096)])
def test_weight_dequant_ragged(fp8, shape):
    codes = syn.random_e4m3_codes(shape, 21)
    s = syn.random_scales(((shape[0] + 127) // 128, (shape[1] + 127) // 128), 22)
    y = fp8.fp8_weight_dequant(dev_e4m3(codes), dev_f32(s))
    assert np.array_equal(host_bits(y), oracle.weight_dequant(codes, s))


@pytest.mark.parametrize("ue8m0", [False, True])
def test_silu_mul_quant(fp8, ue8m0):
    R, I = 300, 1024
    rng = np.random.default_rng(8)
    h13 = syn.to_bf16_bits((2.0 * rng.standard_normal((R, 2 * I))).astype(np.float32))
    h13[3, :128] = 0                                # g block of zeros
    t = dev_bf16(h13)
    y, s, g = fp8.fp8_silu_mul_quant(t, t[:, I:], 2 * I, R, I,
                                     fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32, want_g=True)
    g_gpu = host_bits(g)
    g_ref = oracle.silu_mul(h13[:, :I], h13[:, I:])
    gv, rv = oracle.bf16_to_f32(g_gpu).astype(np.float64), oracle.bf16_to_f32(g_ref).astype(np.float64)
    # fp32 silu on the GPU vs exact silu: a bf16 rounding of silu can flip
    # (one ulp), which moves the product by at most ~2 ulps; rare.
    assert np.all(np.abs(gv - rv) <= 2.0 ** -6 * np.abs(rv) + 1e-30)
    assert np.mean(g_gpu != g_ref) < 2e-3
    # stage-wise: the quantisation of the GPU's own g is bit-exact
    yo, so = oracle.act_quant(g_gpu, ue8m0=ue8m0)
    assert np.array_equal(host_f32(s), so)
    assert np.array_equal(host_bits(y), yo)


def _decision_point_blocks(seed, n_blocks):
    """Blocks whose quotients x/s land on, and within a few fp32 ulps of,
    every e4m3 rounding decision point (midpoints between neighbouring e4m3
    values, incl. the subnormal ones and 2^-10) for varied scales."""
    rng = np.random.default_rng(seed)
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)                       # 0 .. 448
    mids = np.concatenate([(vals[:-1] + vals[1:]) / 2.0, [2.0 ** -10]])
    rows = []
    for _ in range(n_blocks):
        amax = float(np.exp2(rng.uniform(-8, 8)))
        amax = float(syn.bf16_bits_to_f32(syn.to_bf16_bits(np.array([amax], np.float32)))[0])
        s = np.float32(np.float32(amax) / np.float32(448.0))
        tgt = rng.choice(mids, size=127) * float(s) * (1.0 + rng.integers(-6, 7, size=127) * 2.0 ** -23)
        tgt *= np.where(rng.random(127) < 0.5, -1.0, 1.0)
        blk = np.concatenate([[amax], tgt]).astype(np.float32)
        rows.append(blk)
    x = np.stack(rows).reshape(n_blocks // 8, 8 * 128)
    return syn.to_bf16_bits(x)


def test_act_quant_at_rounding_decision_points(fp8):
    # bf16 inputs cannot hit every midpoint exactly, but the rounding to bf16
    # scatters them densely around the decision points of each block's scale
    x = _decision_point_blocks(17, 4096)
    _act_case(fp8, x, False)
    _act_case(fp8, x, True)


def _division_domain_blocks():
    """Every (block-max mantissa, value mantissa, exponent gap 0..-22, sign)
    combination: x / s for s = RN(amax / 448) is determined by these alone
    (fp32 rounding is scale-free in the normal range and gaps below -22 give
    code 0), plus every bf16 value below the 1e-4 floor against the floored
    scale.  Returned as bf16 bit patterns [rows, 1024] (8 blocks per row)."""
    m = np.arange(128, dtype=np.uint32)
    blocks = []
    for am in m:                                   # block max = (1 + am/128) * 2^0
        amax_bits = np.uint16(0x3F80 | am)
        vals = []
        for gap in range(0, 23):
            exp_field = 127 - gap
            for sgn in (0, 0x8000):
                vals.append((sgn | (exp_field << 7) | m).astype(np.uint16))
        vals = np.concatenate(vals)
        amax_f = syn.bf16_bits_to_f32(np.array([amax_bits], np.uint16))[0]
        vals = vals[np.abs(syn.bf16_bits_to_f32(vals)) <= amax_f]
        for i in range(0, len(vals), 127):
            chunk = vals[i:i + 127]
            blk = np.zeros(128, dtype=np.uint16)
            blk[0] = amax_bits
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
    # floored blocks: every positive and negative bf16 below 1e-4
    small = np.arange(0, 0x38D1, dtype=np.uint32).astype(np.uint16)      # 0 .. just below 1e-4
    small = small[syn.bf16_bits_to_f32(small) < 1e-4]
    small = np.concatenate([small, small | np.uint16(0x8000)])
    for i in range(0, len(small), 128):
        blk = np.zeros(128, dtype=np.uint16)
        chunk = small[i:i + 128]
        blk[:len(chunk)] = chunk
        blocks.append(blk)
    blocks = np.stack(blocks)
    pad = (-len(blocks)) % 8
    if pad:
        blocks = np.concatenate([blocks, np.zeros((pad, 128), np.uint16)])
    return blocks.reshape(-1, 8 * 128)


def test_act_quant_division_domain_exhaustive(fp8):
    _act_case(fp8, _division_domain_blocks(), False)


def _every_block_max_blocks(seed):
    """One 128-block per finite bf16 magnitude (+0 .. 0x7F7F as bit
    patterns), that magnitude being the block's max |x| (random sign and
    position); the other 127 values are random bf16 no larger in magnitude,
    random signs.  Returned as bf16 bit patterns [rows, 128]."""
    rng = np.random.default_rng(seed)
    mags = np.arange(0, 0x7F80, dtype=np.int64)
    n = len(mags)
    others = (rng.random((n, 127)) * (mags[:, None] + 1)).astype(np.int64)
    signs = rng.integers(0, 2, size=(n, 128)).astype(np.int64) << 15
    x = np.empty((n, 128), dtype=np.int64)
    pos = rng.integers(0, 128, size=n)
    x[:, :127] = others
    x[:, 127] = mags
    idx = np.arange(128)[None, :]
    x = np.where(idx == pos[:, None], mags[:, None], np.where(idx < pos[:, None], x, np.roll(x, 1, axis=1)))
    return (x | signs).astype(np.uint16)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_act_quant_scale_for_every_bf16_block_max(fp8, ue8m0):
    # the scale RN(max(amax, 1e-4) / 448) on its whole domain: every finite
    # bf16 magnitude is the max of one block; scales and codes bit-exact
    _act_case(fp8, _every_block_max_blocks(61 + ue8m0), ue8m0)
