"""GPU parity of the w1|w3 products with the expert body fused into their
epilogue (behavior-traces page, "MoE trace": w2(silu(w1 x) * w3 x); source
tour, "FP8 with per-block scales" and "Honest Limits": the quantised input
of w2, a fused grouped GEMM instead of the per-expert loop).

fp8_gemm_swiglu and fp8_moe_expert_up (after fp8_moe_quant_scatter) must produce, bit for
bit, the codes and scales of the unfused chain -- fp8_gemm / fp8_act_quant +
fp8_moe_gather + fp8_grouped_gemm with bf16 outputs, then
fp8_silu_mul_quant -- whose stages
the other parity tests check against the oracle.  Shapes are chosen so that
the unfused GEMM also runs whole tiles (the same fp32 summation order).  On
top, sampled rows of g are checked against the oracle's chain (exact GEMM,
bf16 rounding, silu*mul) within the rounding of h and of the codes."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import dev_bf16, dev_e4m3, dev_f32, dev_i32, host_bits, host_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _weights(fp8, I, K, seed, fmt, G=None):
    lead = () if G is None else (G,)
    w1 = syn.normal_bf16_device(lead + (I, K), 0.02, seed, "cuda")
    w3 = syn.normal_bf16_device(lead + (I, K), 0.02, seed + 1, "cuda")
    qs = []
    for w in (w1, w3):
        if G is None:
            qs.append(fp8.fp8_weight_quant(w, fmt))
        else:
            q = torch.empty(lead + (I, K), dtype=torch.float8_e4m3fn, device="cuda")
            s = torch.empty(lead + (I // 128, K // 128), dtype=torch.float32, device="cuda")
            for g in range(G):
                fp8.fp8_weight_quant(w[g], fmt, q=q[g], s=s[g])
            qs.append((q, s))
    (q1, s1), (q3, s3) = qs
    plain = (torch.cat([q1.view(torch.uint8), q3.view(torch.uint8)], -2).contiguous().view(torch.float8_e4m3fn),
             torch.cat([s1, s3], -2).contiguous())
    inter = (fp8.interleave_w13(q1, q3), fp8.interleave_w13(s1, s3, block=1))
    return plain, inter


def _oracle_rows(aq, as_, w1q, w1s, w3q, w3s, rows, ue8m0):
    """The oracle's chain on sampled rows: exact h1, h3 rounded to bf16, then
    silu*mul and act_quant."""
    r1, _ = oracle.gemm(aq, as_, w1q, w1s, rows=rows)
    r3, _ = oracle.gemm(aq, as_, w3q, w3s, rows=rows)
    h1 = oracle.f32_to_bf16(r1.astype(np.float32))
    h3 = oracle.f32_to_bf16(r3.astype(np.float32))
    g = oracle.silu_mul(h1, h3)
    return g, oracle.act_quant(g, ue8m0=ue8m0)


def _check_against_oracle(gq, gs, g_ref):
    """Dequantised codes against the oracle's g: within e4m3 rounding (and
    the rare 1-ulp differences of h, hence of g)."""
    deq = oracle.e4m3_decode(gq).astype(np.float64) * np.repeat(gs.astype(np.float64), 128, axis=1)
    gv = oracle.bf16_to_f32(g_ref).astype(np.float64)
    step = np.repeat(gs.astype(np.float64), 128, axis=1)
    err = np.abs(deq - gv)
    assert np.all(err <= 2.0 ** -3 * np.abs(gv) + 2.0 ** -6 * step), "fused g differs from the oracle's chain"


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
@pytest.mark.parametrize("shape", [(2051, 4608, 512), (300, 4608, 128)])
def test_dense_swiglu_matches_unfused_chain(fp8, shape, ue8m0):
    M, I, K = shape
    fmt = fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32
    (w13, s13), (w13i, s13i) = _weights(fp8, I, K, 600 + M, fmt)
    x = syn.normal_bf16_device((M, K), 1.0, 610 + M, "cuda")
    aq, as_ = fp8.fp8_act_quant(x, fmt)
    # unfused: h = a w13^T (bf16), then silu*mul+act_quant
    assert fp8.fp8_gemm_workspace_size(M, 2 * I, K) == 0    # whole tiles: the same summation order
    h = fp8.fp8_gemm(aq, as_, w13, s13, out_bf16=True)[0]
    yq, ys, _ = fp8.fp8_silu_mul_quant(h, h[:, I:], 2 * I, M, I, fmt)
    gq, gs = fp8.fp8_gemm_swiglu(aq, as_, w13i, s13i, fmt)
    fp8.fp8_device_status()
    assert np.array_equal(host_f32(gs).view(np.uint32), host_f32(ys).view(np.uint32)), "scales differ"
    assert np.array_equal(host_bits(gq), host_bits(yq)), "codes differ"
    rows = np.unique(np.r_[0, 1, 127, 128, M - 1, np.random.default_rng(M).integers(0, M, 3)])
    aq_h, as_h = host_bits(aq), host_f32(as_)
    w_h, s_h = host_bits(w13), host_f32(s13)
    g_ref, _ = _oracle_rows(aq_h, as_h, w_h[:I], s_h[:I // 128], w_h[I:], s_h[I // 128:], rows, ue8m0)
    _check_against_oracle(host_bits(gq)[rows], host_f32(gs)[rows], g_ref)


@pytest.mark.parametrize("ue8m0", [False, True], ids=["fp32", "ue8m0"])
def test_moe_expert_up_matches_unfused_chain(fp8, ue8m0):
    # 700 tokens x top-4 of 16 experts (Zipf): experts with no rows, with
    # fewer than 128 and with several 128-row tiles
    T, E, topk, I, K = 700, 16, 4, 1024, 1024
    fmt = fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32
    rt = syn.moe_routing(T=T, E=E, topk=topk, seed=syn.SEED_BASE + 21)
    ids = rt.ids.copy()
    cold = int(rt.expert_perm[-1])
    for t in np.nonzero((ids == cold).any(axis=1))[0]:    # the coldest expert gets no row
        free = [e for e in range(E) if e != cold and e not in ids[t]]
        ids[t][ids[t] == cold] = free[0]
    assert np.all(np.sort(ids, axis=1)[:, 1:] != np.sort(ids, axis=1)[:, :-1]), "duplicate expert in a token"
    (w13, s13), (w13i, s13i) = _weights(fp8, I, K, 620, fmt, G=E)
    x = syn.normal_bf16_device((T, K), 1.0, 630, "cuda")
    off, pr, rtok = fp8.fp8_moe_route(dev_i32(ids), E)
    xq, xs = fp8.fp8_act_quant(x, fmt)
    # unfused: gather, grouped w1|w3 (bf16), silu*mul+act_quant
    aq, as_ = fp8.fp8_moe_gather(xq, xs, rtok)
    h = fp8.fp8_grouped_gemm(aq, as_, w13, s13, off, out_bf16=True)[0]
    R = T * topk
    yq, ys, _ = fp8.fp8_silu_mul_quant(h, h[:, I:], 2 * I, R, I, fmt)
    # fused: act_quant + gather in one pass, then the grouped w1|w3 with the
    # expert body in its epilogue
    aq2, as2 = fp8.fp8_moe_quant_scatter(x, pr, fmt)
    gq, gs = fp8.fp8_moe_expert_up(aq2, as2, w13i, s13i, off, fmt)
    fp8.fp8_device_status()
    assert np.array_equal(host_bits(aq2), host_bits(aq)), "quant_scatter codes differ from act_quant + gather"
    assert np.array_equal(host_f32(as2).view(np.uint32), host_f32(as_).view(np.uint32)), "quant_scatter scales"
    offs = off.cpu().numpy()
    counts = np.diff(offs)
    assert counts.min() == 0 and counts.max() > 128 and np.any((counts > 0) & (counts < 128))
    assert np.array_equal(host_f32(gs).view(np.uint32), host_f32(ys).view(np.uint32)), "scales differ"
    assert np.array_equal(host_bits(gq), host_bits(yq)), "codes differ"
    # sampled packed rows against the oracle (each row with its expert's weights)
    rtok_h = rtok.cpu().numpy()
    xq_h, xs_h = host_bits(xq), host_f32(xs)
    w_h, s_h = host_bits(w13), host_f32(s13)
    rng = np.random.default_rng(7)
    for r in rng.choice(R, 6, replace=False):
        e = int(np.searchsorted(offs, r, side="right") - 1)
        t = int(rtok_h[r])
        g_ref, _ = _oracle_rows(xq_h[t:t + 1], xs_h[t:t + 1], w_h[e, :I], s_h[e, :I // 128], w_h[e, I:],
                                s_h[e, I // 128:], None, ue8m0)
        _check_against_oracle(host_bits(gq)[r:r + 1], host_f32(gs)[r:r + 1], g_ref)
