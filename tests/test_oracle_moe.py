"""Pins of the oracle's MoE pieces: routing to packed expert rows, the
expert body's silu(h1)*h3, and the weighted scatter-add of expert outputs
(behavior-traces page, "MoE trace": y[idx] += expert(x[idx]) * weight).
"""
import numpy as np
import pytest
import torch

import synthetic as syn


def test_route_is_a_stable_counting_sort(orc):
    rt = syn.moe_routing(T=300, E=16, topk=4, seed=5)
    offsets, pair_row, row_token = orc.moe_route(rt.ids, 16)
    counts = np.bincount(rt.ids.reshape(-1), minlength=16)
    assert np.array_equal(np.diff(offsets), counts) and offsets[0] == 0
    assert np.array_equal(np.sort(pair_row.reshape(-1)), np.arange(1200))
    T, K = rt.ids.shape
    for t in range(T):
        for j in range(K):
            r = pair_row[t, j]
            e = rt.ids[t, j]
            assert offsets[e] <= r < offsets[e + 1]
            assert row_token[r] == t
    # brute force of the stable order inside each expert
    for e in range(16):
        pairs = [p for p in range(T * K) if rt.ids.reshape(-1)[p] == e]
        assert list(pair_row.reshape(-1)[pairs]) == list(range(offsets[e], offsets[e + 1]))


def test_routing_generator_has_distinct_experts_per_token():
    rt = syn.moe_routing(T=512, E=32, topk=8, seed=6)
    for row in rt.ids:
        assert len(set(row.tolist())) == 8
    assert np.allclose(rt.weights.sum(axis=1), 2.5, rtol=1e-6)
    assert np.all(rt.weights > 0)


def test_combine_brute_force_and_one_hot(orc):
    rng = np.random.default_rng(1)
    T, K, D = 6, 3, 5
    R = T * K
    out = syn.to_bf16_bits(rng.standard_normal((R, D)).astype(np.float32))
    pair_row = rng.permutation(R).astype(np.int32).reshape(T, K)
    w = rng.random((T, K)).astype(np.float32)
    y, ymag = orc.moe_combine(out, w, pair_row)
    of = syn.bf16_bits_to_f32(out).astype(np.float64)
    for t in range(T):
        want = sum(float(w[t, j]) * of[pair_row[t, j]] for j in range(K))
        assert np.allclose(y[t], want, rtol=0, atol=1e-15)
        wmag = sum(abs(float(w[t, j]) * of[pair_row[t, j]]) for j in range(K))
        assert np.allclose(ymag[t], wmag, rtol=0, atol=1e-15)
    onehot = np.zeros((T, K), np.float32)
    onehot[:, 1] = 1.0
    y1, _ = orc.moe_combine(out, onehot, pair_row)
    assert np.array_equal(y1, of[pair_row[:, 1]])
    ys, _ = orc.moe_combine(out, w, pair_row, tokens=[4, 1])
    assert np.array_equal(ys, y[[4, 1]])


def test_silu_mul_against_library(orc):
    rng = np.random.default_rng(2)
    h1 = syn.to_bf16_bits((3 * rng.standard_normal(200000)).astype(np.float32))
    h3 = syn.to_bf16_bits(rng.standard_normal(200000).astype(np.float32))
    g = orc.silu_mul(h1, h3)
    t1 = torch.from_numpy(h1.view(np.int16)).view(torch.bfloat16)
    t3 = torch.from_numpy(h3.view(np.int16)).view(torch.bfloat16)
    lib = (torch.nn.functional.silu(t1) * t3).view(torch.int16).numpy().view(np.uint16)
    gf = syn.bf16_bits_to_f32(g).astype(np.float64)
    lf = syn.bf16_bits_to_f32(lib).astype(np.float64)
    # torch computes silu in fp32; the oracle in double.  They may differ by a
    # bf16 ulp of silu, which moves the product by at most ~2 ulps, rarely.
    diff = np.abs(gf - lf)
    assert np.mean(g != lib) < 2e-3
    assert np.all(diff <= 2.0 ** -6 * np.abs(gf) + 1e-30)


def test_silu_mul_special_values(orc):
    f = np.array([0.0, -0.0, 30.0, -30.0, 1.0], np.float32)
    h1 = syn.to_bf16_bits(f)
    h3 = syn.to_bf16_bits(np.array([2.0, 2.0, 0.5, 1.0, 1.0], np.float32))
    g = syn.bf16_bits_to_f32(orc.silu_mul(h1, h3))
    assert g[0] == 0.0 and g[1] == 0.0
    assert g[2] == 15.0                      # silu(30) rounds to 30 in bf16
    assert abs(g[3]) < 1e-10                 # silu(-30) ~ -2.8e-12
    # silu(1) = 1/(1+e^-1) = 0.7310585..., bf16 -> 0.73046875
    assert g[4] == 0.73046875
