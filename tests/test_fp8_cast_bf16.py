"""The offline FP8 -> BF16 conversion (behavior-traces page, bullet
"fp8->bf16 trace"): host-side logic on the CPU -- the safetensors container
round trip and the plan (which tensors are dequantised, passed through with
a warning, kept or dropped; the pruned index) -- and, on the GPU, the whole
conversion of a synthetic three-shard checkpoint checked tensor by tensor
against the oracle's weight_dequant, bit for bit."""
import json
import os
from collections import OrderedDict

import numpy as np
import pytest
import torch

import oracle
import synthetic as syn
from fp8_block_scaled_07_gb300 import fp8_cast_bf16 as conv


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_container_round_trip(tmp_path):
    rng = np.random.default_rng(1)
    t = OrderedDict()
    t["a.weight"] = torch.from_numpy(rng.integers(0, 256, (3, 32), dtype=np.uint8)).view(torch.float8_e4m3fn)
    t["a.weight_scale_inv"] = torch.from_numpy(rng.random((1, 1), dtype=np.float32))
    t["b.bias"] = _bf16(syn.normal_bf16(rng, (5,)))
    t["c.ids"] = torch.arange(7, dtype=torch.int64)
    t["d.scalar"] = torch.tensor(2.5, dtype=torch.float32)
    t["e.empty"] = torch.zeros((0, 4), dtype=torch.float32)
    p = str(tmp_path / "x.safetensors")
    conv.save_file(t, p, {"format": "pt"})
    hdr, meta, base = conv.read_header(p)
    assert meta == {"format": "pt"} and base % 8 == 0
    assert hdr["a.weight"]["dtype"] == "F8_E4M3" and hdr["b.bias"]["dtype"] == "BF16"
    back = conv.load_file(p)
    assert list(back) == list(t)
    for k in t:
        assert back[k].dtype == t[k].dtype and tuple(back[k].shape) == tuple(t[k].shape)
        assert torch.equal(back[k].view(torch.uint8) if back[k].dtype == torch.float8_e4m3fn else back[k],
                           t[k].view(torch.uint8) if t[k].dtype == torch.float8_e4m3fn else t[k])


def test_plan_dequantises_e4m3_with_scales_and_prunes_the_index():
    weight_map = OrderedDict([
        ("l0.wq.weight", "m-1.safetensors"), ("l0.wq.weight_scale_inv", "m-2.safetensors"),
        ("l0.norm.weight", "m-1.safetensors"),
        ("l1.wo.weight", "m-2.safetensors"), ("l1.wo.weight_scale_inv", "m-2.safetensors"),
        ("l1.orphan.weight", "m-2.safetensors"),              # e4m3 without a scale
        ("l1.mask", "m-3.safetensors"),                         # a one-byte tensor that is not e4m3
    ])
    files = {
        "m-2.safetensors": OrderedDict([("l0.wq.weight_scale_inv", "F32"), ("l1.wo.weight", "F8_E4M3"),
                                        ("l1.wo.weight_scale_inv", "F32"), ("l1.orphan.weight", "F8_E4M3")]),
        "m-1.safetensors": OrderedDict([("l0.wq.weight", "F8_E4M3"), ("l0.norm.weight", "BF16")]),
        "m-3.safetensors": OrderedDict([("l1.mask", "U8")]),
    }
    plan, new_map = conv.conversion_plan(weight_map, files)
    assert [f for f, _ in plan] == ["m-1.safetensors", "m-2.safetensors", "m-3.safetensors"]
    acts = dict(plan)
    assert acts["m-1.safetensors"] == [("l0.wq.weight", "dequant", "l0.wq.weight_scale_inv"),
                                       ("l0.norm.weight", "keep", None)]
    assert acts["m-2.safetensors"] == [("l1.wo.weight", "dequant", "l1.wo.weight_scale_inv"),
                                       ("l1.orphan.weight", "passthrough_no_scale", "l1.orphan.weight_scale_inv")]
    assert acts["m-3.safetensors"] == [("l1.mask", "keep", None)]
    assert list(new_map) == ["l0.wq.weight", "l0.norm.weight", "l1.wo.weight", "l1.orphan.weight", "l1.mask"]
    assert new_map["l1.wo.weight"] == "m-2.safetensors"


def _write_checkpoint(root):
    """Three shards: wq_a (7168 cols) whose scale lives in the next shard, a
    ragged wkv_a (576 rows) and a bf16 norm, an e4m3 tensor with no scale."""
    rng = np.random.default_rng(syn.SEED_BASE + 12)
    wa = syn.normal_bf16(rng, (1536, 7168), 0.02)
    wk = syn.normal_bf16(rng, (576, 7168), 0.02)
    qa, sa = oracle.weight_quant(wa)
    qk, sk = oracle.weight_quant(wk)
    orphan = rng.integers(0, 0x7F, (128, 256), dtype=np.uint8)
    norm = syn.normal_bf16(rng, (7168,), 1.0)
    f8 = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn)
    shards = {
        "model-00001-of-00003.safetensors": OrderedDict([("layers.0.attn.wq_a.weight", f8(qa)),
                                                         ("layers.0.attn_norm.weight", _bf16(norm))]),
        "model-00002-of-00003.safetensors": OrderedDict([("layers.0.attn.wq_a.weight_scale_inv", torch.from_numpy(sa)),
                                                         ("layers.0.attn.wkv_a.weight", f8(qk)),
                                                         ("layers.0.attn.wkv_a.weight_scale_inv", torch.from_numpy(sk))]),
        "model-00003-of-00003.safetensors": OrderedDict([("layers.0.orphan.weight", f8(orphan))]),
    }
    wm = OrderedDict()
    for fname, tensors in shards.items():
        conv.save_file(tensors, os.path.join(root, fname), {"format": "pt"})
        for k in tensors:
            wm[k] = fname
    with open(os.path.join(root, conv.INDEX_NAME), "w") as f:
        json.dump({"metadata": {"total_size": 0}, "weight_map": wm}, f)
    return {"layers.0.attn.wq_a.weight": (qa, sa), "layers.0.attn.wkv_a.weight": (qk, sk)}, orphan, norm


@pytest.mark.gpu
def test_conversion_of_a_synthetic_checkpoint(tmp_path):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    src, dst = tmp_path / "fp8", tmp_path / "bf16"
    os.makedirs(src)
    weights, orphan, norm = _write_checkpoint(str(src))
    warnings = []
    names = conv.fp8_cast_bf16(str(src), str(dst), log=warnings.append)
    assert sorted(names) == sorted(weights)
    assert len(warnings) == 1 and "layers.0.orphan.weight" in warnings[0]
    with open(dst / conv.INDEX_NAME) as f:
        index = json.load(f)
    assert not any(k.endswith("_scale_inv") for k in index["weight_map"])
    assert index["weight_map"]["layers.0.attn.wkv_a.weight"] == "model-00002-of-00003.safetensors"
    out = {}
    for fname in sorted(os.listdir(dst)):
        if fname.endswith(".safetensors"):
            for k, v in conv.load_file(str(dst / fname)).items():
                assert not k.endswith("_scale_inv")
                out[k] = v
    for name, (q, s) in weights.items():
        got = out[name]
        assert got.dtype == torch.bfloat16
        want = oracle.weight_dequant(q, s)
        assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), want), name
    assert np.array_equal(out["layers.0.orphan.weight"].view(torch.uint8).numpy(), orphan)
    assert np.array_equal(out["layers.0.attn_norm.weight"].view(torch.int16).numpy().view(np.uint16), norm)
