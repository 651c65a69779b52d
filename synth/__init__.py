"""Seeded synthetic inputs for the W4A16 GEMV workloads.

This module is the one thing the oracle side (tests) and the GPU side (bench,
smoke, tests) share.  It draws random numbers and describes the workload
shapes; it holds none of the method's arithmetic (no quantisation, packing,
unpacking or dot products).

Recipe.  Weights W[N][K] ~ Normal(0, std = 0.02) in fp32; activations
x[M][K] ~ Normal(0, 1) rounded to fp16.  The numbers come from torch's seeded
generator on the device that is asked for: the CPU generator (Mersenne
Twister) and the CUDA generator (Philox) give different streams for the same
seed, so every parity test draws on the CPU and uploads; the bench draws its
large weight sets on the GPU, where only timing depends on them.

The pages measure real Qwen2.5-Coder-7B checkpoints; these seeded tensors of
the same shapes stand in for them (no checkpoint is needed to time or check a
GEMV).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

W_STD = 0.02
GROUP = 128

# Qwen2.5-7B-shaped decoder layer: hidden 3584, 28 query heads and 4 KV heads
# of dimension 128 (KV width 512), FFN width 18944, 28 layers.
HIDDEN = 3584
KV_DIM = 512
FFN = 18944
N_LAYERS = 28

# projection index inside a layer (also the order of the per-layer seeds)
PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


def proj_shape(name: str, hidden: int = HIDDEN, kv_dim: int = KV_DIM, ffn: int = FFN):
    """(N, K) of one projection's weight, nn.Linear convention (out x in)."""
    return {
        "q": (hidden, hidden),
        "k": (kv_dim, hidden),
        "v": (kv_dim, hidden),
        "o": (hidden, hidden),
        "gate": (ffn, hidden),
        "up": (ffn, hidden),
        "down": (hidden, ffn),
    }[name]


def layer_seed(layer: int, proj: int) -> int:
    """Seed of projection `proj` (0..6, PROJ_NAMES order) of layer `layer`;
    proj == 7 is that layer's activation vector."""
    return 1000 + 8 * layer + proj


@dataclass(frozen=True)
class Gemv:
    """One GEMV workload: y[M][N] = x[M][K] . W[N][K]^T."""
    name: str
    M: int
    N: int
    K: int
    seed: int
    group: int = GROUP


# The five workloads.  Configs 1 and 3 are families of GEMVs.
TINY = Gemv("tiny", 1, 512, 1024, 0)
Q_PROJ = Gemv("q_proj", 1, HIDDEN, HIDDEN, 1)
KV_PROJ = Gemv("kv_proj", 1, KV_DIM, HIDDEN, 2)
GATE_UP = Gemv("gate_up", 1, 2 * FFN, HIDDEN, 3)
DOWN_SWEEP = tuple(Gemv(f"down_m{m}", m, HIDDEN, FFN, 4) for m in (1, 2, 4, 8, 16))
ALL_GEMVS = (TINY, Q_PROJ, KV_PROJ, GATE_UP) + DOWN_SWEEP


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weights(N: int, K: int, seed: int, device="cpu", std: float = W_STD) -> torch.Tensor:
    """fp32 W[N][K] ~ Normal(0, std)."""
    g = _gen(seed, device)
    return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * std


def activations(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """fp16 x[M][K] ~ Normal(0, 1), drawn in fp32 and rounded to fp16.
    Uses a stream distinct from the weights' stream of the same seed."""
    g = _gen(seed * 7919 + 17, device)
    return torch.randn((M, K), generator=g, device=device, dtype=torch.float32).to(torch.float16)


def gemv_inputs(cfg: Gemv, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """(W fp32 [N][K], x fp16 [M][K]) for one workload."""
    return weights(cfg.N, cfg.K, cfg.seed, device), activations(cfg.M, cfg.K, cfg.seed, device)


def uniform_ints(shape, low: int, high: int, seed: int, device="cpu") -> torch.Tensor:
    """Integers uniform in [low, high) (int64), for hand-built test patterns."""
    g = _gen(seed, device)
    return torch.randint(low, high, shape, generator=g, device=device, dtype=torch.int64)
