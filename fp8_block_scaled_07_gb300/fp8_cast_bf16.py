"""Offline FP8 -> BF16 checkpoint conversion on the GPU's weight_dequant.

What it does follows the behavior-traces page ("Behavior traces --
deepseek-ai/DeepSeek-V3", bullet "fp8->bf16 trace") and the data-flow page
(bullet on fp8_cast_bf16): read the checkpoint's ``model.safetensors.index.json``
weight map to find every tensor across the shard files, take the shard files
in sorted order, and for each file

  * drop the ``*_scale_inv`` entries (the block scales),
  * dequantise every e4m3 tensor ``name`` with its scale grid
    ``name + "_scale_inv"`` (which may live in another shard file; the last
    two files loaded stay cached on the device) through
    :func:`fp8_block_scaled_07_gb300.fp8_weight_dequant`, and pass the tensor
    through unchanged, with a warning, when it has no scale,
  * keep every other tensor as it is,

write the file under the same name, and finally write an index whose weight
map has lost the ``*_scale_inv`` keys.

Readings where the pages leave a step open: "each 1-byte tensor" is taken
as "each tensor of safetensors dtype F8_E4M3" (other one-byte dtypes, e.g.
U8 or BOOL, pass through); every ``*_scale_inv`` key leaves the index, since
every shard file drops those entries.

The safetensors container is read and written by this module itself (an
8-byte little-endian header length, a JSON header naming each tensor's dtype,
shape and byte range, then the raw little-endian data): the format, not a
library.  The dequantisation runs in the library's CUDA kernel; there is no
CPU path.
"""
import json
import os
import struct
import sys
from collections import OrderedDict

import numpy as np
import torch

INDEX_NAME = "model.safetensors.index.json"
SCALE_SUFFIX = "_scale_inv"

# safetensors dtype name -> (torch dtype, bytes per element)
DTYPES = {
    "F8_E4M3": (torch.float8_e4m3fn, 1),
    "BF16": (torch.bfloat16, 2),
    "F16": (torch.float16, 2),
    "F32": (torch.float32, 4),
    "F64": (torch.float64, 8),
    "I64": (torch.int64, 8),
    "I32": (torch.int32, 4),
    "I16": (torch.int16, 2),
    "I8": (torch.int8, 1),
    "U8": (torch.uint8, 1),
    "BOOL": (torch.bool, 1),
}
_NAMES = {v[0]: k for k, v in DTYPES.items()}


# ------------------------------------------------------------------ container
def read_header(path):
    """-> (header dict without __metadata__, metadata dict, data offset)."""
    with open(path, "rb") as f:
        (n,) = struct.unpack("<Q", f.read(8))
        hdr = json.loads(f.read(n).decode("utf-8"))
    meta = hdr.pop("__metadata__", {}) or {}
    return hdr, meta, 8 + n


def load_file(path, device="cpu"):
    """All tensors of a safetensors file -> OrderedDict name -> tensor (in
    the file's header order), moved to `device`."""
    hdr, _, base = read_header(path)
    raw = np.fromfile(path, dtype=np.uint8)
    out = OrderedDict()
    for name, info in hdr.items():
        dt, size = DTYPES[info["dtype"]]
        b, e = info["data_offsets"]
        shape = tuple(info["shape"])
        n = int(np.prod(shape)) if shape else 1
        if e - b != n * size:
            raise ValueError(f"{path}: {name}: byte range does not match its shape and dtype")
        if n == 0:
            t = torch.empty(shape, dtype=dt)
        else:
            t = torch.from_numpy(raw[base + b:base + e].copy()).view(dt).reshape(shape)
        out[name] = t.to(device) if device != "cpu" else t
    return out


def save_file(tensors, path, metadata=None):
    """Write name -> tensor (contiguous, any of DTYPES) as a safetensors file."""
    hdr, blobs, off = {}, [], 0
    for name, t in tensors.items():
        t = t.detach().contiguous().cpu()
        if t.dtype not in _NAMES:
            raise TypeError(f"{name}: dtype {t.dtype} has no safetensors name here")
        nbytes = t.numel() * t.element_size()
        hdr[name] = {"dtype": _NAMES[t.dtype], "shape": list(t.shape), "data_offsets": [off, off + nbytes]}
        blobs.append(t.reshape(-1).view(torch.uint8).numpy() if nbytes else np.zeros(0, np.uint8))
        off += nbytes
    if metadata:
        hdr["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    h = json.dumps(hdr, separators=(",", ":")).encode("utf-8")
    h += b" " * ((8 - len(h) % 8) % 8)   # the data starts 8-byte aligned
    tmp = path + ".tmp"
    with open(tmp, "wb") as f:
        f.write(struct.pack("<Q", len(h)))
        f.write(h)
        for blob in blobs:
            f.write(blob.tobytes())
    os.replace(tmp, path)


# ------------------------------------------------------------------ plan
def conversion_plan(weight_map, file_dtypes):
    """Host-side decisions of the conversion, per shard file in sorted order.

    weight_map: tensor name -> shard file name (the index's weight map);
    file_dtypes: shard file name -> OrderedDict tensor name -> safetensors
    dtype.  Returns (plan, new_weight_map) where plan is a list of
    (file, [(name, action, scale_name)]) with action "dequant" (an e4m3
    tensor with a scale), "passthrough_no_scale" (an e4m3 tensor whose scale
    is missing) or "keep"; scale tensors are left out (dropped)."""
    plan = []
    for fname in sorted(file_dtypes):
        acts = []
        for name, dt in file_dtypes[fname].items():
            if name.endswith(SCALE_SUFFIX):
                continue
            if dt == "F8_E4M3":
                sname = name + SCALE_SUFFIX
                acts.append((name, "dequant" if sname in weight_map else "passthrough_no_scale", sname))
            else:
                acts.append((name, "keep", None))
        plan.append((fname, acts))
    new_map = OrderedDict((k, v) for k, v in weight_map.items() if not k.endswith(SCALE_SUFFIX))
    return plan, new_map


# ------------------------------------------------------------------ driver
class _FileCache:
    """The last `size` shard files loaded, on the device."""

    def __init__(self, root, device, size=2):
        self.root, self.device, self.size = root, device, size
        self.files = OrderedDict()

    def get(self, fname):
        if fname in self.files:
            self.files.move_to_end(fname)
            return self.files[fname]
        state = load_file(os.path.join(self.root, fname), self.device)
        self.files[fname] = state
        while len(self.files) > self.size:
            self.files.popitem(last=False)
        return state


def fp8_cast_bf16(input_dir, output_dir, device="cuda", log=None):
    """Convert the FP8 checkpoint in `input_dir` to BF16 in `output_dir`.
    Returns the list of tensor names that were dequantised."""
    import fp8_block_scaled_07_gb300 as fp8

    log = log or (lambda msg: print(msg, file=sys.stderr))
    os.makedirs(output_dir, exist_ok=True)
    with open(os.path.join(input_dir, INDEX_NAME)) as f:
        index = json.load(f)
    weight_map = index["weight_map"]
    shard_files = sorted(n for n in os.listdir(input_dir) if n.endswith(".safetensors"))
    file_dtypes = {}
    for fname in shard_files:
        hdr, _, _ = read_header(os.path.join(input_dir, fname))
        file_dtypes[fname] = OrderedDict((k, v["dtype"]) for k, v in hdr.items())
    plan, new_map = conversion_plan(weight_map, file_dtypes)
    cache = _FileCache(input_dir, device)
    converted = []
    for fname, acts in plan:
        state = cache.get(fname)
        _, meta, _ = read_header(os.path.join(input_dir, fname))
        out = OrderedDict()
        for name, action, sname in acts:
            t = state[name]
            if action == "dequant":
                s = cache.get(weight_map[sname])[sname]
                if t.dim() != 2 or s.dim() != 2:
                    raise ValueError(f"{name}: weight_dequant takes 2-D tensors")
                out[name] = fp8.fp8_weight_dequant(t, s.to(torch.float32).contiguous())
                converted.append(name)
            else:
                if action == "passthrough_no_scale":
                    log(f"fp8_cast_bf16: warning: no {sname} for {name}; written unchanged")
                out[name] = t
        if device != "cpu":
            torch.cuda.synchronize()
        save_file(out, os.path.join(output_dir, fname), meta)
        # the cache keeps state for later scale lookups; the outputs go
        del out
    new_index = {"metadata": index.get("metadata", {}), "weight_map": new_map}
    with open(os.path.join(output_dir, INDEX_NAME), "w") as f:
        json.dump(new_index, f, indent=2)
    return converted


def main(argv=None):
    import argparse
    ap = argparse.ArgumentParser(description="FP8 (e4m3 + 128x128 scales) -> BF16 checkpoint conversion")
    ap.add_argument("--input-fp8-hf-path", required=True)
    ap.add_argument("--output-bf16-hf-path", required=True)
    a = ap.parse_args(argv)
    names = fp8_cast_bf16(a.input_fp8_hf_path, a.output_bf16_hf_path)
    print(f"dequantised {len(names)} tensors")


if __name__ == "__main__":
    main()
