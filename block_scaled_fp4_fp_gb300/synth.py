"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module holds random-number generation and shape bookkeeping only -- none of
the quantization or matmul arithmetic.  Every tensor is drawn with an explicit
``torch.Generator`` seed so the CUDA path and the CPU oracle see identical bits.

Workload shapes (the pages' decode and prefill shapes):
  * decode stack: hidden 5120, MLP 17408, 64 layers, projections q/k/v/o
    (5120x5120), gate/up (17408x5120), down (5120x17408), weights ~ N(0, 0.02);
  * activations ~ N(0, 1), optionally with 0.1 % outliers scaled by 50;
  * MoE: 32 experts, top-4 routing, 2048 tokens, hidden 2880, gate/up 5760.
"""
from __future__ import annotations

import numpy as np
import torch

HIDDEN = 5120
MLP = 17408
LAYERS = 64
# (name, N rows, K cols) for one decoder layer; W is stored [N, K].
LAYER_PROJECTIONS = (
    ("q", HIDDEN, HIDDEN),
    ("k", HIDDEN, HIDDEN),
    ("v", HIDDEN, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", MLP, HIDDEN),
    ("up", MLP, HIDDEN),
    ("down", HIDDEN, MLP),
)

MOE_EXPERTS = 32
MOE_TOPK = 4
MOE_TOKENS = 2048
MOE_HIDDEN = 2880
MOE_GATE_UP = 5760


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std: float = 1.0, seed: int = 0, device="cpu") -> torch.Tensor:
    """bf16(std * N(0, 1)) drawn in fp32 with a seeded generator."""
    g = _gen(seed, device)
    t = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def activations_with_outliers(rows: int, cols: int, seed: int = 0, outlier_seed: int = 1,
                              frac: float = 1e-3, mult: float = 50.0, device="cpu") -> torch.Tensor:
    """bf16 N(0,1) activations where elements with rand < frac are scaled by ``mult``."""
    g = _gen(seed, device)
    t = torch.randn((rows, cols), generator=g, dtype=torch.float32, device=device)
    g2 = _gen(outlier_seed, device)
    mask = torch.rand((rows, cols), generator=g2, dtype=torch.float32, device=device) < frac
    t = torch.where(mask, t * mult, t)
    return t.to(torch.bfloat16)


def layer_seed(layer: int, proj: int) -> int:
    """Seed of projection ``proj`` (index into LAYER_PROJECTIONS) of ``layer``."""
    return 1000 * layer + proj


def moe_routing(tokens: int = MOE_TOKENS, experts: int = MOE_EXPERTS, topk: int = MOE_TOPK,
                seed: int = 0):
    """Uniform top-k routing: rand(tokens, experts).topk(k) gives distinct experts
    per token; routed rows are stably sorted by expert.  Returns (lhs, rhs) int32
    arrays of length tokens*topk: lhs = token index, rhs = expert index."""
    g = _gen(seed, "cpu")
    scores = torch.rand((tokens, experts), generator=g)
    experts_of = scores.topk(topk, dim=1).indices  # [tokens, topk]
    rhs = experts_of.reshape(-1).to(torch.int64)
    lhs = torch.arange(tokens).repeat_interleave(topk)
    order = torch.sort(rhs, stable=True).indices
    return (lhs[order].to(torch.int32).numpy().copy(), rhs[order].to(torch.int32).numpy().copy())


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (copied to host)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def from_u16(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)


# ------------------------------------------------------------- decode stack
def layer_groups(layout: str):
    """The GEMVs of one decode layer as (N, K, projection indices stacked as
    rows): "split" is one matrix per projection, "fused_qkv" stores q|k|v as one
    matrix, "fused" stores q|k|v and gate|up as one each (the projections that
    multiply the same x)."""
    projs = LAYER_PROJECTIONS
    groups = {"split": [[p] for p in range(len(projs))],
              "fused_qkv": [[0, 1, 2], [3], [4], [5], [6]],
              "fused": [[0, 1, 2], [3], [4, 5], [6]]}
    if layout not in groups:
        raise ValueError(layout)
    out = []
    for grp in groups[layout]:
        assert len({projs[p][2] for p in grp}) == 1, "stacked projections share K"
        out.append((sum(projs[p][1] for p in grp), projs[grp[0]][2], grp))
    return out


def decode_weight(layer: int, grp, device="cpu") -> torch.Tensor:
    """bf16 weights of one GEMV of the decode stack: the projections of ``grp``
    (indices into LAYER_PROJECTIONS) drawn as bf16(0.02 N(0, 1)) with their own
    seeds and stacked as rows."""
    parts = [bf16_normal((LAYER_PROJECTIONS[p][1], LAYER_PROJECTIONS[p][2]), 0.02, seed=layer_seed(layer, p),
                         device=device) for p in grp]
    return parts[0] if len(parts) == 1 else torch.cat(parts)


def decode_x(K: int, device="cpu") -> torch.Tensor:
    """The decode stack's activation vector for inputs of width K: bf16 N(0, 1)."""
    return bf16_normal((K,), 1.0, seed=7 + K, device=device)


def affine_synthetic(N: int, K: int, seed: int, group: int = 64, device="cpu"):
    """Synthetic affine-4 weights of the decode stack: uniform random packed
    codes (int32 [N, K/8]) and per-group bf16 scale and bias drawn around the
    range an affine quantizer gives for N(0, 0.02) groups (scale ~ 0.11/15,
    bias ~ -0.055).  Returns (codes, scales, biases)."""
    g = _gen(seed, device)
    q = torch.randint(-2 ** 31, 2 ** 31 - 1, (N, K // 8), generator=g, device=device, dtype=torch.int64)
    q = q.to(torch.int32)
    s = (0.11 / 15 * (1 + 0.1 * torch.rand((N, K // group), generator=g, device=device))).to(torch.bfloat16)
    b = (-0.055 * (1 + 0.1 * torch.rand((N, K // group), generator=g, device=device))).to(torch.bfloat16)
    return q, s, b
