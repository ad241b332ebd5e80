"""Seeded synthetic inputs shaped like DeepSeek-V3's FP8 linears.

This module draws random numbers and nothing else: it holds none of the
quantisation or GEMM arithmetic.  It feeds both the CUDA library and the CPU
oracle, which therefore see identical inputs.  bf16 tensors are returned as
``np.uint16`` bit patterns (host path) or ``torch.bfloat16`` tensors (device
path, for sizes the host cannot draw quickly).

Recipe (one numpy ``PCG64`` stream per tensor, spawned from a per-workload
``SeedSequence``):
  * activations ~ N(0, 1), a fixed fraction of entries (chosen without
    replacement) multiplied by an outlier factor;
  * weights ~ N(0, 0.02);
  * values are drawn in float32 and rounded to bf16 (round to nearest even,
    by torch's conversion);
  * MoE routing: expert ranks r = 1..E get probability proportional to 1/r
    (Zipf, s = 1) over a seeded permutation of the experts; each token draws
    top-k distinct experts by sequential sampling without replacement; gate
    logits ~ N(0, 1) become sigmoid weights normalised over the token's
    experts and multiplied by the route scale (the gate's output, which the
    linear layer consumes as data).
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

SEED_BASE = 1000

# Layer shapes (N = out features, K = in features) of the DeepSeek-V3 671B
# projections used by the workloads.
DECODE_LAYERS: Dict[str, Tuple[int, int]] = {
    "wq_a": (1536, 7168),
    "wq_b": (24576, 1536),
    "wo": (7168, 16384),
}
MLP_DIM, MLP_INTER = 7168, 18432
MOE_DIM, MOE_INTER, MOE_EXPERTS, MOE_TOPK, MOE_ROUTE_SCALE = 7168, 2048, 256, 8, 2.5
WKV_A = (576, 7168)
DEQUANT_SHAPE = (18432, 7168)


def _streams(seed: int, n: int) -> List[np.random.Generator]:
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (RNE) through torch's conversion."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_f32(rng: np.random.Generator, shape, std=1.0, outlier_frac=0.0,
               outlier_mult=1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if outlier_frac > 0.0:
        n = int(round(outlier_frac * x.size))
        if n:
            pos = rng.choice(x.size, size=n, replace=False)
            flat = x.reshape(-1)
            flat[pos] *= np.float32(outlier_mult)
    return x


def normal_bf16(rng, shape, std=1.0, outlier_frac=0.0, outlier_mult=1.0) -> np.ndarray:
    return to_bf16_bits(normal_f32(rng, shape, std, outlier_frac, outlier_mult))


def normal_bf16_device(shape, std, seed: int, device="cuda", outlier_frac=0.0,
                       outlier_mult=1.0):
    """Device-side draw (torch Philox) for tensors too large to draw on the
    host; same distribution as :func:`normal_bf16`."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if outlier_frac > 0.0:
        n = int(round(outlier_frac * x.numel()))
        if n:
            pos = torch.randperm(x.numel(), generator=g, device=device)[:n]
            x.view(-1)[pos] *= outlier_mult
    return x.to(torch.bfloat16)


# ------------------------------------------------------------------ workloads
@dataclass
class Linear:
    """One linear layer's inputs: activations x [M, K], weight w [N, K]."""
    name: str
    x: np.ndarray
    w: np.ndarray
    ue8m0: bool = False


def tiny_linear(seed=SEED_BASE + 0) -> Linear:
    """4 tokens x 256 -> 256, 1% outliers x20."""
    rx, rw = _streams(seed, 2)
    x = normal_bf16(rx, (4, 256), 1.0, 0.01, 20.0)
    w = normal_bf16(rw, (256, 256), 0.02)
    return Linear("tiny", x, w)


def decode_linears(M=16, seed=SEED_BASE + 1, layers=None) -> List[Linear]:
    """wq_a / wq_b / wo at batch M, activations with 0.5% outliers x30."""
    names = list(DECODE_LAYERS) if layers is None else list(layers)
    rs = _streams(seed + 17 * M, 2 * len(DECODE_LAYERS))
    out = []
    for i, name in enumerate(DECODE_LAYERS):
        if name not in names:
            continue
        N, K = DECODE_LAYERS[name]
        x = normal_bf16(rs[2 * i], (M, K), 1.0, 0.005, 30.0)
        w = normal_bf16(rs[2 * i + 1], (N, K), 0.02)
        out.append(Linear(name, x, w))
    return out


def decode_activations(M, K, seed) -> np.ndarray:
    (r,) = _streams(seed, 1)
    return normal_bf16(r, (M, K), 1.0, 0.005, 30.0)


def mlp_activations(M=4096, K=MLP_DIM, seed=SEED_BASE + 2) -> np.ndarray:
    (r,) = _streams(seed, 1)
    return normal_bf16(r, (M, K), 1.0)


def mlp_weight(name: str, shape, seed=SEED_BASE + 2) -> np.ndarray:
    idx = {"w1": 1, "w3": 2, "w2": 3}[name]
    rs = _streams(seed, 4)
    return normal_bf16(rs[idx], shape, 0.02)


@dataclass
class Routing:
    ids: np.ndarray       # int32 [T, topk], distinct per row
    weights: np.ndarray   # float32 [T, topk]
    expert_perm: np.ndarray


def moe_routing(T=4096, E=MOE_EXPERTS, topk=MOE_TOPK, seed=SEED_BASE + 3,
                route_scale=MOE_ROUTE_SCALE) -> Routing:
    r_perm, r_pick, r_logit = _streams(seed, 3)
    perm = r_perm.permutation(E)
    p = np.zeros(E, dtype=np.float64)
    p[perm] = 1.0 / np.arange(1, E + 1, dtype=np.float64)     # rank r -> 1/r
    p /= p.sum()
    P = np.tile(p, (T, 1))
    ids = np.empty((T, topk), dtype=np.int32)
    rows = np.arange(T)
    for j in range(topk):                                     # sequential, w/o replacement
        cdf = np.cumsum(P, axis=1)
        u = r_pick.random(T) * cdf[:, -1]
        pick = (cdf < u[:, None]).sum(axis=1)
        pick = np.minimum(pick, E - 1)
        # guard against landing on an already-taken (zero-mass) expert at a
        # cdf plateau: step to the next expert that still has mass
        while True:
            bad = P[rows, pick] == 0.0
            if not bad.any():
                break
            pick[bad] = (pick[bad] + 1) % E
        ids[:, j] = pick
        P[rows, pick] = 0.0
    logits = r_logit.standard_normal(size=(T, topk))
    sig = 1.0 / (1.0 + np.exp(-logits))
    w = (sig / sig.sum(axis=1, keepdims=True) * route_scale).astype(np.float32)
    return Routing(ids, w, perm)


def moe_activations(T=4096, K=MOE_DIM, seed=SEED_BASE + 3) -> np.ndarray:
    rs = _streams(seed + 101, 1)
    return normal_bf16(rs[0], (T, K), 1.0)


def moe_expert_weight_device(expert: int, which: str, seed=SEED_BASE + 3, device="cuda"):
    """Expert weights are drawn on the device (256 experts x 3 matrices)."""
    idx = {"w1": 0, "w3": 1, "w2": 2}[which]
    shape = (MOE_INTER, MOE_DIM) if which in ("w1", "w3") else (MOE_DIM, MOE_INTER)
    return normal_bf16_device(shape, 0.02, seed * 1_000_003 + expert * 3 + idx, device)


def moe_expert_weight_host(expert: int, which: str, N: int, K: int, seed=SEED_BASE + 3):
    """Host draw of one expert's weight, for small grouped-GEMM cases."""
    idx = {"w1": 0, "w3": 1, "w2": 2}[which]
    (r,) = _streams(seed * 1_000_003 + expert * 3 + idx, 1)
    return normal_bf16(r, (N, K), 0.02)


def ragged_ue8m0(M=37, seed=SEED_BASE + 4) -> Linear:
    """wkv_a (7168 -> 576, last N block half full), scale_fmt ue8m0, with
    injected special 128-blocks: x row 0 block 0 all zero; x row 1 block 1
    constant +1.5; x last row, last block constant -7.25; W block (0,0) all
    zero; W last (partial) block constant 0.03125."""
    N, K = WKV_A
    rx, rw = _streams(seed + 31 * M, 2)
    x = normal_f32(rx, (M, K), 1.0, 0.005, 30.0)
    w = normal_f32(rw, (N, K), 0.02)
    x[0, 0:128] = 0.0
    if M > 1:
        x[1, 128:256] = 1.5
    x[M - 1, K - 128:K] = -7.25
    w[0:128, 0:128] = 0.0
    nb_last = (N - 1) // 128
    w[nb_last * 128:N, K - 128:K] = 0.03125
    return Linear("wkv_a", to_bf16_bits(x), to_bf16_bits(w), ue8m0=True)


def dequant_source(shape=DEQUANT_SHAPE, seed=SEED_BASE + 4) -> np.ndarray:
    """bf16 weight whose quantised form is the weight_dequant input."""
    (r,) = _streams(seed + 7, 1)
    return normal_bf16(r, shape, 0.02)


def uniform_bf16(shape, lo, hi, seed) -> np.ndarray:
    (r,) = _streams(seed, 1)
    return to_bf16_bits(r.uniform(lo, hi, size=shape).astype(np.float32))


def random_e4m3_codes(shape, seed) -> np.ndarray:
    """Uniformly random finite e4m3 codes (NaN codes 0x7F/0xFF excluded)."""
    (r,) = _streams(seed, 1)
    c = r.integers(0, 256, size=shape, dtype=np.uint8)
    nan = (c & 0x7F) == 0x7F
    c[nan] = c[nan] - 1
    return c


def random_pow2_scales(shape, seed, lo=-12, hi=4) -> np.ndarray:
    """Positive power-of-two fp32 scales (the ue8m0 scale format), exponents in [lo, hi)."""
    (r,) = _streams(seed, 1)
    return np.exp2(r.integers(lo, hi, size=shape)).astype(np.float32)


def random_scales(shape, seed, lo=-12, hi=4) -> np.ndarray:
    """Positive fp32 scales with a spread of exponents and full mantissas."""
    (r,) = _streams(seed, 1)
    m = r.uniform(1.0, 2.0, size=shape)
    e = r.integers(lo, hi, size=shape)
    return (m * np.exp2(e)).astype(np.float32)
