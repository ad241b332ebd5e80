"""Launch ordering on one stream: every kernel of the library lets the next
one start early (programmatic dependent launch) and waits for earlier
launches only where it first touches global memory.  A call that reads
buffers the previous kernel is still writing must see the new data: here
fp8_weight_quant (which lets its dependents start at once) writes fresh
weights and block scales, and the GEMM reading them is launched right after
it with no host synchronisation.  Each result must equal, bit for bit, the
same call made after a full synchronisation."""
import numpy as np
import pytest
import torch

import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import fp8_block_scaled_07_gb300 as m
    return m


def _chained_vs_settled(fp8, call, N, K, rounds=4):
    wq = torch.empty((N, K), dtype=torch.float8_e4m3fn, device="cuda")
    ws = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device="cuda")
    weights = [syn.normal_bf16_device((N, K), 0.02, 500 + i, "cuda") for i in range(rounds)]
    torch.cuda.synchronize()
    chained, kept = [], []
    for i in range(rounds):
        fp8.fp8_weight_quant(weights[i], q=wq, s=ws)   # writes the buffers the next call reads
        chained.append(call(wq, ws).clone())
        kept.append((wq.clone(), ws.clone()))
    torch.cuda.synchronize()
    fp8.fp8_device_status()
    for i, (q, s) in enumerate(kept):
        torch.cuda.synchronize()
        settled = call(q, s)
        torch.cuda.synchronize()
        assert torch.equal(chained[i].view(torch.int16), settled.view(torch.int16)), f"round {i}: stale inputs read"
    fp8.fp8_device_status()


@pytest.mark.parametrize("layer", ["wq_a", "wq_b", "wo"])
def test_fused_decode_linear_reads_fresh_weights(fp8, layer):
    N, K = syn.DECODE_LAYERS[layer]
    x = syn.normal_bf16_device((16, K), 1.0, 510, "cuda")
    _chained_vs_settled(fp8, lambda q, s: fp8.fp8_linear(x, q, s)[0], N, K)


def test_staged_linear_reads_fresh_weights(fp8):
    N, K = syn.DECODE_LAYERS["wq_a"]
    x = syn.normal_bf16_device((48, K), 1.0, 511, "cuda")
    _chained_vs_settled(fp8, lambda q, s: fp8.fp8_linear(x, q, s)[0], N, K)


@pytest.mark.parametrize("M", [16, 512])
def test_gemm_reads_fresh_weights(fp8, M):
    # swapped decode schedule (M=16) and the dense prefill schedule (M=512)
    N, K = 2048, 2048
    xq, xs = fp8.fp8_act_quant(syn.normal_bf16_device((M, K), 1.0, 512 + M, "cuda"))
    _chained_vs_settled(fp8, lambda q, s: fp8.fp8_gemm(xq, xs, q, s)[0], N, K)


@pytest.mark.parametrize("M", [16, 64, 256])
def test_gemm_reads_activations_quantised_just_before(fp8, M):
    # act_quant writes the codes and scales fp8_gemm reads next, round after
    # round (the decode kernel at M = 16 and 64, the dense one at M = 256)
    N, K = 1024, 2048
    w, w_s = fp8.fp8_weight_quant(syn.normal_bf16_device((N, K), 0.02, 520, "cuda"))
    xq = torch.empty((M, K), dtype=torch.float8_e4m3fn, device="cuda")
    xs = torch.empty((M, K // 128), dtype=torch.float32, device="cuda")
    xs_in = [syn.normal_bf16_device((M, K), 1.0, 521 + i, "cuda") for i in range(4)]
    torch.cuda.synchronize()
    chained = []
    for x in xs_in:
        fp8.fp8_act_quant(x, y=xq, s=xs)
        chained.append(fp8.fp8_gemm(xq, xs, w, w_s)[0].clone())
    torch.cuda.synchronize()
    for i, x in enumerate(xs_in):
        q, s = fp8.fp8_act_quant(x)
        torch.cuda.synchronize()
        settled = fp8.fp8_gemm(q, s, w, w_s)[0]
        torch.cuda.synchronize()
        assert torch.equal(chained[i].view(torch.int16), settled.view(torch.int16)), f"round {i}: stale inputs read"
    fp8.fp8_device_status()


def test_linear_reads_activations_written_just_before(fp8):
    # weight_dequant writes the bf16 activations the fused decode linear
    # quantises next, round after round
    M, N, K = 16, 1536, 7168
    w, w_s = fp8.fp8_weight_quant(syn.normal_bf16_device((N, K), 0.02, 530, "cuda"))
    src = [fp8.fp8_weight_quant(syn.normal_bf16_device((M, K), 1.0, 531 + i, "cuda")) for i in range(4)]
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    chained = []
    for q, s in src:
        fp8.fp8_weight_dequant(q, s, y=x)
        chained.append(fp8.fp8_linear(x, w, w_s)[0].clone())
    torch.cuda.synchronize()
    for i, (q, s) in enumerate(src):
        xi = fp8.fp8_weight_dequant(q, s)
        torch.cuda.synchronize()
        settled = fp8.fp8_linear(xi, w, w_s)[0]
        torch.cuda.synchronize()
        assert torch.equal(chained[i].view(torch.int16), settled.view(torch.int16)), f"round {i}: stale inputs read"
    fp8.fp8_device_status()


def test_query_projection_chain(fp8):
    # wq_a -> wq_b at a decode batch, as a decoder chains them (minus the
    # norm in between): the second fused linear quantises the first one's
    # bf16 output, launched right behind it, round after round with one
    # output buffer.  Each round must equal the settled chain bit for bit and
    # match the oracle's chain (exact GEMM, bf16 rounding, act_quant, GEMM).
    import oracle
    from tests.helpers import check_gemm, host_bits, host_f32

    M = 16
    (Na, Ka), (Nb, Kb) = syn.DECODE_LAYERS["wq_a"], syn.DECODE_LAYERS["wq_b"]
    wa, wa_s = fp8.fp8_weight_quant(syn.normal_bf16_device((Na, Ka), 0.02, 540, "cuda"))
    wb, wb_s = fp8.fp8_weight_quant(syn.normal_bf16_device((Nb, Kb), 0.02, 541, "cuda"))
    xs = [syn.normal_bf16_device((M, Ka), 1.0, 542 + i, "cuda") for i in range(3)]
    ya = torch.empty((M, Na), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    chained = []
    for x in xs:
        fp8.fp8_linear(x, wa, wa_s, c_bf16=ya)
        chained.append(fp8.fp8_linear(ya, wb, wb_s, out_fp32=True))
    torch.cuda.synchronize()
    fp8.fp8_device_status()
    wa_h, wa_sh, wb_h, wb_sh = host_bits(wa), host_f32(wa_s), host_bits(wb), host_f32(wb_s)
    for i, x in enumerate(xs):
        y1 = fp8.fp8_linear(x, wa, wa_s)[0]
        torch.cuda.synchronize()
        sb, sf = fp8.fp8_linear(y1, wb, wb_s, out_fp32=True)
        torch.cuda.synchronize()
        cb, cf = chained[i]
        assert torch.equal(cb.view(torch.int16), sb.view(torch.int16)), f"round {i}: stale activations read"
        assert torch.equal(cf.view(torch.int32), sf.view(torch.int32)), f"round {i}: stale activations read"
        # the oracle's chain from the same first-layer output
        aq, as_ = oracle.act_quant(host_bits(y1))
        ref, mag = oracle.gemm(aq, as_, wb_h, wb_sh)
        check_gemm(ref, mag, host_f32(cf), host_bits(cb), f"round {i}: wq_b after wq_a")
    fp8.fp8_device_status()
