"""Pins of the oracle's act_quant / weight quantisation / weight_dequant.

What fixes them (source tour, "FP8 with per-block scales"; data-flow page,
"FP8 quantization data flow"): one fp32 scale per 128-element block equal to
the clamped block max over 448; codes are the e4m3 roundings of x/scale.
Pins: hand-derived worked blocks (tests/golden), zero and constant blocks,
the block max always landing on the e4m3 ceiling, the e4m3 round-trip error
bound, ue8m0 scales being the next power of two, and a composition of
library routines (torch's own fp8 conversion) as an independent codec.
"""
import json
import os

import numpy as np
import pytest
import torch

import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLOOR = np.float32(1e-4)


def _f32(h):
    return syn.bf16_bits_to_f32(h)


def test_golden_worked_blocks(orc):
    with open(os.path.join(GOLDEN, "act_quant_worked_blocks.json")) as f:
        data = json.load(f)
    for case in data["cases"]:
        x = np.zeros((1, 128), dtype=np.uint16)
        lead = [int(h, 16) for h in case["x_bf16"]]
        x[0, :len(lead)] = lead
        # the bit patterns are the values they claim to be
        assert np.array_equal(_f32(x[0, :len(lead)]).astype(np.float64),
                              np.array(case["x_values"], dtype=np.float64))
        y, s = orc.act_quant(x, ue8m0=case["ue8m0"])
        assert s.shape == (1, 1)
        assert float(s[0, 0]) == case["scale"], case["name"]
        want = np.zeros(128, dtype=np.uint8)
        codes = [int(h, 16) for h in case["codes"]]
        want[:len(codes)] = codes
        assert np.array_equal(y[0], want), case["name"]


def test_zero_block_uses_the_floor(orc):
    x = np.zeros((3, 256), dtype=np.uint16)
    x[1, 128:] = syn.to_bf16_bits(np.linspace(-2, 2, 128, dtype=np.float32))
    y, s = orc.act_quant(x)
    floor_scale = np.float32(FLOOR / np.float32(448.0))
    assert s[0, 0] == floor_scale and s[0, 1] == floor_scale and s[1, 0] == floor_scale
    assert s[1, 1] == np.float32(np.float32(2.0) / np.float32(448.0))
    assert not y[0].any() and not y[1, :128].any()


def test_negative_zero_block(orc):
    x = np.full((1, 128), 0x8000, dtype=np.uint16)
    y, s = orc.act_quant(x)
    assert np.all(y == 0x80)


@pytest.mark.parametrize("c", [1.5, -7.25, 0.03125, 300.0, -1e-3, 3e-5])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_constant_block(orc, c, ue8m0):
    x = np.full((2, 128), syn.to_bf16_bits(np.array([c], np.float32))[0], dtype=np.uint16)
    y, s = orc.act_quant(x, ue8m0=ue8m0)
    cv = float(_f32(x[0, :1])[0])
    vals = orc.e4m3_decode(y)
    assert np.all(y == y[0, 0])
    if abs(cv) >= 1e-4:
        if not ue8m0:
            assert abs(vals[0, 0]) == 448.0
        else:
            assert 224.0 <= abs(vals[0, 0]) <= 448.0
    assert np.sign(vals[0, 0]) == np.sign(cv) or vals[0, 0] == 0


def _act_inputs(M, K, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-12, 8, size=(M, K // 128, 1))).repeat(128, axis=2).reshape(M, K)
    out = rng.random((M, K)) < 0.01
    x[out] *= 30
    return syn.to_bf16_bits(x)


@pytest.mark.parametrize("ue8m0", [False, True])
def test_block_max_hits_the_ceiling_and_roundtrip_bound(orc, ue8m0):
    x = _act_inputs(37, 1024, 1)
    y, s = orc.act_quant(x, ue8m0=ue8m0)
    xf = _f32(x).astype(np.float64).reshape(37, 8, 128)
    q = orc.e4m3_decode(y).reshape(37, 8, 128)
    sc = s.astype(np.float64)[:, :, None]
    amax = np.abs(xf).max(axis=2)
    imax = np.abs(xf).argmax(axis=2)
    top = np.abs(np.take_along_axis(q, imax[:, :, None], axis=2))[:, :, 0]
    if not ue8m0:
        assert np.all(top == 448.0)
        assert np.array_equal(s, (np.maximum(amax, 1e-4).astype(np.float32) / np.float32(448)))
    else:
        m, e = np.frexp(s)
        assert np.all(m == 0.5)
        raw = np.maximum(amax, 1e-4).astype(np.float32) / np.float32(448)
        assert np.all(s >= raw) and np.all(s / 2 < raw)
        assert np.all((top >= 224.0) & (top <= 448.0))
    # e4m3 round trip: relative 2^-4 in the normal range, absolute 2^-10 * s below it
    err = np.abs(q * sc - xf)
    normal = np.abs(xf) / sc >= 2.0 ** -6
    slack = 1 + 2.0 ** -20
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]) * slack)
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(sc, xf.shape)[~normal] * slack)


def test_matches_composition_of_library_routines(orc):
    x = _act_inputs(64, 2048, 2)
    y, s = orc.act_quant(x)
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().view(64, 16, 128)
    amax = xt.abs().amax(dim=2).clamp(min=1e-4)
    st = amax / 448.0
    yt = (xt / st[:, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).reshape(64, 2048)
    assert np.array_equal(s, st.numpy())
    assert np.array_equal(y, yt.numpy())


def test_weight_quant_blocks_and_partial_edges(orc):
    rng = np.random.default_rng(4)
    N, K = 300, 384                      # 3 N-blocks (last has 44 rows), 3 K-blocks
    w = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    w[0:128, 0:128] = 0.0                # zero block
    w[256:300, 256:384] = 0.03125        # constant partial block
    w[290, 10] = 5.0                     # max of block (2, 0) lies in the partial rows
    wb = syn.to_bf16_bits(w)
    q, s = orc.weight_quant(wb)
    assert s.shape == (3, 3)
    wf = _f32(wb).astype(np.float64)
    vals = orc.e4m3_decode(q)
    for nb in range(3):
        for kb in range(3):
            blk = wf[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = max(np.abs(blk).max(), 1e-4)
            assert s[nb, kb] == np.float32(np.float32(amax) / np.float32(448))
            qb = vals[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            if np.abs(blk).max() > 0:
                assert np.abs(qb).max() == 448.0
    assert not q[0:128, 0:128].any()
    assert np.all(q[256:300, 256:384] == 0x7E)
    assert q[290, 10] == 0x7E
    # row-blocks of the weight: same codes as act_quant when one 128x128 block
    # has its max in every row (scales coincide)
    wr = np.tile(syn.to_bf16_bits(rng.standard_normal(128).astype(np.float32)), (128, 1))
    qa, sa = orc.act_quant(wr)
    qw, sw = orc.weight_quant(wr)
    assert np.array_equal(qa, qw) and np.all(sa == sw[0, 0])


def test_weight_dequant_unit_scale_is_the_decoded_code(orc):
    codes = np.arange(256, dtype=np.uint8).reshape(2, 128)
    codes[codes == 0x7F] = 0x7E
    codes[codes == 0xFF] = 0xFE
    y = orc.weight_dequant(codes, np.ones((1, 1), np.float32))
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(y, lib.numpy().view(np.uint16))


def test_weight_dequant_power_of_two_scales_are_exact(orc):
    codes = syn.random_e4m3_codes((256, 384), 9)
    s = np.exp2(np.arange(-3, 3, dtype=np.float32)).reshape(2, 3)
    y = orc.weight_dequant(codes, s)
    want = orc.e4m3_decode(codes) * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    assert np.array_equal(_f32(y).astype(np.float64), want)


def test_weight_dequant_matches_library_product(orc):
    M, N = 300, 200                               # ragged in both directions
    codes = syn.random_e4m3_codes((M, N), 10)
    s = syn.random_scales((3, 2), 11)
    y = orc.weight_dequant(codes, s)
    wt = torch.from_numpy(codes).view(torch.float8_e4m3fn).float()
    st = torch.from_numpy(s).repeat_interleave(128, 0)[:M].repeat_interleave(128, 1)[:, :N]
    lib = (wt * st).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(y, lib)
