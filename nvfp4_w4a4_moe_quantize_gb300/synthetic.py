"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This module only draws random numbers and casts them to BF16; it contains none of
the NVFP4 or MoE arithmetic.  Every tensor comes from a CPU ``torch.Generator`` with
an explicit seed, so the CUDA path and the CPU oracle receive identical bytes.

Workload shapes follow the Qwen3-30B-A3B expert block that the pages measure on
("The 4-bitter Lesson: Balancing Stability and Performance in NVFP4 RL", §Baseline:
Qwen3-30B-A3B, 8k sequences): hidden 2048, intermediate 768, 128 experts, top-8.
The pages' own data (DAPO-math-17k rollouts, trained weights) is not available, so
Gaussian activations / weights and a Zipf-skewed router stand in for it.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = [
    "MoEShape",
    "WORKLOADS",
    "randn_bf16",
    "outlier_channels_bf16",
    "router_logits_normal",
    "router_logits_zipf",
    "moe_inputs",
    "bf16_bits",
]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, std: float = 1.0, seed: int = 0) -> torch.Tensor:
    """N(0, std^2) values rounded (RNE) to BF16, on the CPU."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def outlier_channels_bf16(rows: int, cols: int, frac: float = 0.01, factor: float = 50.0,
                          seed: int = 0) -> torch.Tensor:
    """N(0,1) matrix with round(frac*cols) seeded columns scaled by ``factor`` before the
    BF16 cast (the standalone-quantiser workload: 1% outlier channels x50)."""
    g = _gen(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    n_out = int(round(frac * cols))
    cols_idx = torch.randperm(cols, generator=g)[:n_out]
    x[:, cols_idx] *= factor
    return x.to(torch.bfloat16)


def router_logits_normal(tokens: int, experts: int, seed: int = 0) -> torch.Tensor:
    """i.i.d. N(0,1) router logits, float32 [tokens, experts]."""
    return torch.randn(tokens, experts, generator=_gen(seed), dtype=torch.float32)


def router_logits_zipf(tokens: int, experts: int, s: float = 1.1, seed: int = 0) -> torch.Tensor:
    """Router logits whose top-k is Plackett-Luce sampling from Zipf(s) expert popularity.

    Expert popularity p_e is proportional to 1/rank^s over a seeded permutation of the
    experts; logits = log p_e + Gumbel(0,1) noise, so taking the top k without
    replacement samples experts in proportion to p_e (Gumbel-top-k).
    """
    g = _gen(seed)
    ranks = torch.randperm(experts, generator=g).to(torch.float64) + 1.0
    logp = -s * torch.log(ranks)
    logp = logp - torch.logsumexp(logp, 0)
    u = torch.rand(tokens, experts, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    gumbel = -torch.log(-torch.log(u))
    return (logp[None, :] + gumbel).to(torch.float32)


def bf16_bits(x: torch.Tensor):
    """The uint16 bit patterns of a BF16 CPU tensor, as a numpy array."""
    assert x.dtype == torch.bfloat16
    return x.contiguous().view(torch.int16).numpy().view("uint16")


@dataclass(frozen=True)
class MoEShape:
    """One MoE expert-block workload (tokens, hidden, intermediate, experts, top-k)."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    routing: str = "zipf"          # "zipf" | "normal"
    x_std: float = 1.0
    w_std: float = 0.02
    zipf_s: float = 1.1
    extra: dict = field(default_factory=dict)


# The workloads: a tiny block for exhaustive checks, the Qwen3-30B-A3B-shaped blocks.
WORKLOADS = {
    "tiny": MoEShape("tiny", T=512, H=256, I=128, E=8, k=2, routing="normal"),
    "gateup": MoEShape("gateup", T=8192, H=2048, I=768, E=128, k=8, routing="zipf"),
    "forward": MoEShape("forward", T=16384, H=2048, I=768, E=128, k=8, routing="zipf"),
    "learner": MoEShape("learner", T=32768, H=2048, I=768, E=128, k=8, routing="normal"),
}
QUANTISER_SHAPE = (16384, 2048)


def moe_inputs(shape: MoEShape, seed: int = 0):
    """Seeded inputs for an expert block: x [T,H], router logits [T,E] fp32,
    W13 [E, 2I, H] (gate rows then up rows) and W2 [E, H, I], all BF16 on the CPU.

    Sub-seeds are derived per tensor so that any one tensor can be regenerated alone.
    """
    T = shape.T
    x = randn_bf16((T, shape.H), shape.x_std, seed * 1000 + 1)
    if shape.routing == "zipf":
        logits = router_logits_zipf(T, shape.E, shape.zipf_s, seed * 1000 + 2)
    else:
        logits = router_logits_normal(T, shape.E, seed * 1000 + 2)
    w13 = randn_bf16((shape.E, 2 * shape.I, shape.H), shape.w_std, seed * 1000 + 3)
    w2 = randn_bf16((shape.E, shape.H, shape.I), shape.w_std, seed * 1000 + 4)
    return x, logits, w13, w2


def zipf_expected_rows(shape: MoEShape) -> list:
    """Not used by the path; documents the skew of the Zipf workload (expected rows/expert)."""
    ranks = [r + 1 for r in range(shape.E)]
    w = [1.0 / (r ** shape.zipf_s) for r in ranks]
    z = sum(w)
    return [shape.T * shape.k * wi / z for wi in w]

