"""Seeded synthetic inputs for the MoE layer.

This module only draws random numbers in the shapes and distributions of the
benchmark workloads; it holds none of the layer's arithmetic.  Both the CUDA
path and the CPU oracle consume what it returns.

Recipe (all tensors from one ``torch.Generator`` seeded with ``seed``):
  x    ~ N(0, 1)          [T, H]     -> bf16
  W1   ~ N(0, 0.02^2)     [E, H, I]  -> bf16   (gate)
  W3   ~ N(0, 0.02^2)     [E, H, I]  -> bf16   (up)
  W2   ~ N(0, 0.02^2)     [E, I, H]  -> bf16   (down)
  dout ~ N(0, 1)          [T, H]     -> bf16
  router logits L ~ N(0, 1) [T, E] (float32); the selection key is L + b
  with a per-expert bias b; idx = top-k of the key (columns in descending
  key order), s = softmax over the k chosen *unbiased* logits (float32).

Routing kinds:
  "uniform" b = 0 (uniform load in expectation)
  "zipf"    b_e = log p_(pi(e)), p_r proportional to r^-1.2, pi a seeded
            permutation of the experts (skewed, imbalanced load)
  "hot"     zipf bias, plus: 16 seeded experts get b = -inf (never chosen),
            and a seeded half of the tokens have one expert e* forced into
            their top-k.
"""

from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Shape:
    T: int
    H: int
    I: int
    E: int
    k: int

    @property
    def R(self):
        return self.T * self.k


# Workloads (T, H, I, E, k) and their routing kinds.
WORKLOADS = {
    "tiny": (Shape(256, 256, 128, 8, 2), "uniform", "bf16"),
    "mid": (Shape(4096, 2048, 768, 64, 8), "uniform", "bf16"),
    # small profiling case: weights (~300 MB) still exceed L2, device footprint < 1.5 GB
    "prof": (Shape(2048, 2048, 768, 32, 8), "uniform", "bf16"),
    "dsv3": (Shape(8192, 7168, 2048, 256, 8), "zipf", "bf16"),
    "mid_mxfp8_zipf": (Shape(4096, 2048, 768, 64, 8), "zipf", "mxfp8"),
    "mid_mxfp8_hot": (Shape(4096, 2048, 768, 64, 8), "hot", "mxfp8"),
    "kimi": (Shape(16384, 7168, 2048, 384, 8), "uniform", "bf16"),
    # few experts, long weight-gradient K loops (2,048 routed rows per expert)
    "long_k": (Shape(16384, 7168, 2048, 16, 2), "uniform", "bf16"),
    "kimi_mxfp8": (Shape(16384, 7168, 2048, 384, 8), "uniform", "mxfp8"),
    # small multi-pass ncu cases with the DeepSeek-V3 H and I (weights 1.4 GB,
    # larger than L2; device footprint about 4 GB)
    "prof_wide": (Shape(2048, 7168, 2048, 16, 4), "zipf", "bf16"),
    "prof_wide_mx": (Shape(2048, 7168, 2048, 16, 4), "zipf", "mxfp8"),
}

ZIPF_S = 1.2
HOT_EMPTY_EXPERTS = 16
HOT_TOKEN_FRACTION = 0.5


def _randn(shape, gen, device, std=1.0, chunk_dim0=False):
    if not chunk_dim0:
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    out = torch.empty(shape, device=device, dtype=torch.bfloat16)
    for e in range(shape[0]):
        out[e] = (torch.randn(shape[1:], generator=gen, device=device, dtype=torch.float32) * std).to(torch.bfloat16)
    return out


def routing_bias(E, kind, gen, device):
    """Per-expert selection bias of a routing kind (float32 [E]) and e*."""
    if kind == "uniform":
        return torch.zeros(E, device=device), None
    ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
    p = ranks.pow(-ZIPF_S)
    p = p / p.sum()
    pi = torch.randperm(E, generator=gen, device=device)
    bias = torch.log(p[pi]).to(torch.float32)
    if kind == "zipf":
        return bias, None
    if kind == "hot":
        order = torch.randperm(E, generator=gen, device=device)
        hot = int(order[0])
        empty = order[1:1 + HOT_EMPTY_EXPERTS]
        bias[empty] = -math.inf
        return bias, hot
    raise ValueError(kind)


def make_routing(T, E, k, kind, gen, device):
    logits = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32)
    bias, hot = routing_bias(E, kind, gen, device)
    key = logits + bias
    if hot is not None:
        chosen = torch.randperm(T, generator=gen, device=device)[: int(T * HOT_TOKEN_FRACTION)]
        key[chosen, hot] = math.inf
    _, idx = torch.topk(key, k, dim=1, largest=True, sorted=True)
    chosen_logits = torch.gather(logits, 1, idx)
    s = torch.softmax(chosen_logits, dim=1)
    return idx.to(torch.int32).contiguous(), s.to(torch.float32).contiguous()


def make_inputs(shape: Shape, routing="uniform", seed=0, device="cpu", weights=True):
    """All layer inputs for one workload as a dict of torch tensors."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed))
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    big = E * H * I > (1 << 26)
    out = {}
    out["x"] = _randn((T, H), gen, dev)
    out["idx"], out["s"] = make_routing(T, E, k, routing, gen, dev)
    out["dout"] = _randn((T, H), gen, dev)
    if weights:
        out["W1"] = _randn((E, H, I), gen, dev, 0.02, chunk_dim0=big)
        out["W3"] = _randn((E, H, I), gen, dev, 0.02, chunk_dim0=big)
        out["W2"] = _randn((E, I, H), gen, dev, 0.02, chunk_dim0=big)
    return out


def load_stats(idx, E, tile_rows=128):
    """Realised expert-load statistics of a routing (for reports)."""
    counts = torch.bincount(idx.reshape(-1).long().cpu(), minlength=E)
    padded = int(((counts + tile_rows - 1) // tile_rows * tile_rows).sum())
    return dict(max_rows=int(counts.max()), mean_rows=float(counts.float().mean()),
                empty_experts=int((counts == 0).sum()), padded_rows=padded,
                routed_rows=int(counts.sum()))
