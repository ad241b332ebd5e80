"""GPU parity of the routed-expert path (behavior-traces page, "MoE trace";
source tour, "Honest Limits": a fused grouped GEMM instead of the Python
expert loop): routing to packed rows, gather, the grouped GEMM, the expert
body and the weighted combine."""
import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from tests.helpers import (check_gemm, dev_bf16, dev_e4m3, dev_f32, dev_i32, host_bits,
                           host_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


# T*topk % 4 == 0 takes the 16-byte-load path of the kernel (ragged warp
# ranges included: 4093*8, 1000*2), the others the one-id-per-lane path
# expert groups per CTA: 32 of 32 experts at E = 1024, one CTA at E = 1, a
# last group of one expert at E = 33
@pytest.mark.parametrize("T,E,topk", [(4096, 256, 8), (4093, 256, 8), (1000, 8, 2), (300, 16, 4), (1, 8, 2),
                                      (37, 64, 6), (2000, 1024, 8), (50, 1, 1), (777, 33, 5)])
def test_route_matches_oracle_exactly(fp8, T, E, topk):
    rt = syn.moe_routing(T=T, E=E, topk=topk, seed=T + E)
    off, pr, rtok = fp8.fp8_moe_route(dev_i32(rt.ids), E)
    o_off, o_pr, o_rtok = oracle.moe_route(rt.ids, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    assert np.array_equal(pr.cpu().numpy(), o_pr)
    assert np.array_equal(rtok.cpu().numpy(), o_rtok)


# odd block counts (37 x 3 blocks), topk above 16 (rows read directly past
# the first 16), and the model's shape; both scale formats
@pytest.mark.parametrize("T,K,topk,E", [(37, 384, 6, 16), (5, 128, 20, 32), (300, 7168, 8, 256)])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_quant_scatter_equals_oracle_act_quant_then_gather(fp8, T, K, topk, E, ue8m0):
    rt = syn.moe_routing(T=T, E=E, topk=topk, seed=T + K)
    x = syn.normal_bf16(np.random.default_rng(T), (T, K))
    _, pr, _ = fp8.fp8_moe_route(dev_i32(rt.ids), E)
    aq, as_ = fp8.fp8_moe_quant_scatter(dev_bf16(x), pr, fp8.FP8_SCALE_UE8M0 if ue8m0 else fp8.FP8_SCALE_FP32)
    fp8.fp8_device_status()
    # the oracle: act_quant of every token row, then the packed rows in order
    xq, xs = oracle.act_quant(x, ue8m0=ue8m0)
    _, _, rtok = oracle.moe_route(rt.ids, E)
    assert np.array_equal(host_bits(aq), xq[rtok])
    assert np.array_equal(host_f32(as_).view(np.uint32), xs[rtok].view(np.uint32))


def test_gather_rows(fp8):
    rt = syn.moe_routing(T=300, E=16, topk=4, seed=2)
    x = syn.normal_bf16(np.random.default_rng(1), (300, 512))
    xq, xs = oracle.act_quant(x)
    _, _, rtok = oracle.moe_route(rt.ids, 16)
    aq, as_ = fp8.fp8_moe_gather(dev_e4m3(xq), dev_f32(xs), dev_i32(rtok))
    # gather-then-quantise (the model's order) equals quantise-then-gather
    gq, gs = oracle.act_quant(x[rtok])
    assert np.array_equal(host_bits(aq), gq)
    assert np.array_equal(host_f32(as_), gs)


@pytest.mark.parametrize("topk", [8, 6])
def test_combine(fp8, topk):
    # top-8 (the V3 routing) takes the compile-time path, others the generic one
    T, D = 257, 1024
    rng = np.random.default_rng(3)
    R = T * topk
    out = syn.to_bf16_bits(rng.standard_normal((R, D)).astype(np.float32))
    pair_row = rng.permutation(R).astype(np.int32).reshape(T, topk)
    w = (rng.random((T, topk)) * 0.6).astype(np.float32)
    yb, yf = fp8.fp8_moe_combine(dev_bf16(out), dev_f32(w), dev_i32(pair_row), out_bf16=True, out_fp32=True)
    y, ymag = oracle.moe_combine(out, w, pair_row)
    yf_h = host_f32(yf).astype(np.float64)
    # fp32 sum of topk terms: error below topk * 2^-24 * sum |terms|
    assert np.all(np.abs(yf_h - y) <= topk * 2.0 ** -24 * ymag + 1e-30)
    assert np.array_equal(host_bits(yb), oracle.f32_to_bf16(host_f32(yf)))


def _grouped_case(fp8, G, N, K, counts, seed, rows=None):
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    R = int(offsets[-1]) + 5                   # R_max beyond the routed rows
    a = syn.random_e4m3_codes((R, K), seed)
    as_ = syn.random_scales((R, K // 128), seed + 1)
    b = syn.random_e4m3_codes((G, N, K), seed + 2)
    bs = syn.random_scales((G, (N + 127) // 128, K // 128), seed + 3)
    cb, cf = fp8.fp8_grouped_gemm(dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs), dev_i32(offsets),
                                  out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    ref, mag = oracle.grouped_gemm(a, as_, b, bs, offsets, rows=rows)
    cf_h, cb_h = host_f32(cf), host_bits(cb)
    sel = np.arange(offsets[-1]) if rows is None else np.asarray(rows)
    check_gemm(ref, mag, cf_h[sel], cb_h[sel], f"grouped G={G} N={N} K={K}")


def test_grouped_small_with_empty_and_ragged_groups(fp8):
    _grouped_case(fp8, 6, 256, 384, [0, 5, 130, 0, 257, 1], 11)


def test_grouped_many_groups(fp8):
    rng = np.random.default_rng(4)
    counts = rng.integers(0, 300, 40)
    _grouped_case(fp8, 40, 128, 256, counts, 12)


def test_moe_chain_config_shapes_sampled(fp8):
    """4096 tokens, top-8 of 256 experts (Zipf routing), w1|w3 [2*2048, 7168]
    and w2 [7168, 2048] per expert: each stage checked against the oracle
    fed the previous GPU stage (sampled tokens)."""
    T, E, topk, D, I = 4096, syn.MOE_EXPERTS, syn.MOE_TOPK, syn.MOE_DIM, syn.MOE_INTER
    rt = syn.moe_routing(T=T, E=E, topk=topk)
    x = syn.moe_activations(T=T)
    dev = torch.device("cuda")
    # expert weights drawn on the device, quantised by the library
    w13q = torch.empty((E, 2 * I, D), dtype=torch.float8_e4m3fn, device=dev)
    w13s = torch.empty((E, 2 * I // 128, D // 128), dtype=torch.float32, device=dev)
    w2q = torch.empty((E, D, I), dtype=torch.float8_e4m3fn, device=dev)
    w2s = torch.empty((E, D // 128, I // 128), dtype=torch.float32, device=dev)
    for e in range(E):
        w1 = syn.moe_expert_weight_device(e, "w1")
        w3 = syn.moe_expert_weight_device(e, "w3")
        fp8.fp8_weight_quant(torch.cat([w1, w3], 0), q=w13q[e], s=w13s[e])
        fp8.fp8_weight_quant(syn.moe_expert_weight_device(e, "w2"), q=w2q[e], s=w2s[e])
    ids = dev_i32(rt.ids)
    off, pair_row, row_tok = fp8.fp8_moe_route(ids, E)
    xq, xs = fp8.fp8_act_quant(dev_bf16(x))
    aq, as_ = fp8.fp8_moe_gather(xq, xs, row_tok)
    h13, _ = fp8.fp8_grouped_gemm(aq, as_, w13q, w13s, off)
    gq, gs, g = fp8.fp8_silu_mul_quant(h13, h13[:, I:], 2 * I, T * topk, I, want_g=True)
    o2, _ = fp8.fp8_grouped_gemm(gq, gs, w2q, w2s, off)
    yb, yf = fp8.fp8_moe_combine(o2, dev_f32(rt.weights), pair_row, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()

    o_off, o_pr, o_rtok = oracle.moe_route(rt.ids, E)
    assert np.array_equal(off.cpu().numpy(), o_off)
    tokens = np.array([0, 1, 2047, 4095])
    rows = np.sort(o_pr[tokens].reshape(-1))
    experts = np.unique(rt.ids[tokens])
    # the oracle's own quantisation of the sampled experts' weights
    w13q_h, w13s_h = host_bits(w13q[experts]), host_f32(w13s[experts])
    w2q_h, w2s_h = host_bits(w2q[experts]), host_f32(w2s[experts])
    for k, e in enumerate(experts):
        w1 = syn.moe_expert_weight_device(int(e), "w1").cpu().view(torch.int16).numpy().view(np.uint16)
        w3 = syn.moe_expert_weight_device(int(e), "w3").cpu().view(torch.int16).numpy().view(np.uint16)
        q13, s13 = oracle.weight_quant(np.concatenate([w1, w3], 0))
        assert np.array_equal(q13, w13q_h[k]) and np.array_equal(s13, w13s_h[k])
        w2 = syn.moe_expert_weight_device(int(e), "w2").cpu().view(torch.int16).numpy().view(np.uint16)
        q2, s2 = oracle.weight_quant(w2)
        assert np.array_equal(q2, w2q_h[k]) and np.array_equal(s2, w2s_h[k])
    # stage 1: gather + grouped w1|w3 on the sampled rows (oracle quantises x itself)
    oq, os_ = oracle.act_quant(x[o_rtok[rows]])
    assert np.array_equal(host_bits(aq)[rows], oq)
    sub_off = np.zeros(len(experts) + 1, np.int32)
    row_expert = np.searchsorted(o_off, rows, side="right") - 1
    order = np.argsort(np.searchsorted(experts, row_expert), kind="stable")
    assert np.array_equal(order, np.arange(len(rows)))
    for k, e in enumerate(experts):
        sub_off[k + 1] = sub_off[k] + int(np.sum(row_expert == e))
    ref, mag = oracle.grouped_gemm(oq, os_, w13q_h, w13s_h, sub_off)
    check_gemm(ref, mag, None, host_bits(h13)[rows], "w1|w3")
    # stage 2: expert body on the GPU's h13
    h = host_bits(h13)[rows]
    g_ref = oracle.silu_mul(h[:, :I], h[:, I:])
    g_gpu = host_bits(g)[rows]
    assert np.mean(g_gpu != g_ref) < 2e-3
    qq, qs = oracle.act_quant(g_gpu)
    assert np.array_equal(host_bits(gq)[rows], qq) and np.array_equal(host_f32(gs)[rows], qs)
    # stage 3: grouped w2 on the GPU's g quantisation
    ref2, mag2 = oracle.grouped_gemm(qq, qs, w2q_h, w2s_h, sub_off)
    check_gemm(ref2, mag2, None, host_bits(o2)[rows], "w2")
    # stage 4: combine of the GPU's expert outputs
    y, ymag = oracle.moe_combine(host_bits(o2), rt.weights, o_pr, tokens=tokens)
    yf_h = host_f32(yf)[tokens].astype(np.float64)
    assert np.all(np.abs(yf_h - y) <= topk * 2.0 ** -24 * ymag + 1e-30)


@pytest.mark.parametrize("N", [512, 384])
def test_grouped_bf16_only_tile_store(fp8, N):
    # bf16-only output leaves through 16-row TMA boxes (128x256 tiles for
    # N = 512, 128x128 for 384); an expert's rows ending inside a 16-row half
    # are stored directly.  Bit-identical to the direct stores of a call that
    # also asks for fp32; rows past the last expert keep their sentinel
    counts = [1, 15, 16, 17, 31, 32, 33, 135, 0, 160, 7]
    G, K = len(counts), 256
    offsets = np.zeros(G + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    R = int(offsets[-1]) + 24
    a = syn.random_e4m3_codes((R, K), 21)
    as_ = syn.random_scales((R, K // 128), 22)
    b = syn.random_e4m3_codes((G, N, K), 23)
    bs = syn.random_scales((G, N // 128, K // 128), 24)
    args = (dev_e4m3(a), dev_f32(as_), dev_e4m3(b), dev_f32(bs), dev_i32(offsets))
    sentinel = 0x7FBF
    buf = torch.full((R, N), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    fp8.fp8_grouped_gemm(*args, c_bf16=buf)
    cb, cf = fp8.fp8_grouped_gemm(*args, out_bf16=True, out_fp32=True)
    fp8.fp8_device_status()
    got, ref_b = host_bits(buf), host_bits(cb)
    n = int(offsets[-1])
    assert np.all(got[n:] == sentinel), "rows past the last expert were written"
    assert np.array_equal(got[:n], ref_b[:n]), "TMA-stored bf16 differs from direct stores"
    ref, mag = oracle.grouped_gemm(a, as_, b, bs, offsets)
    check_gemm(ref, mag, host_f32(cf)[:n], got[:n], f"grouped bf16-only N={N}")
