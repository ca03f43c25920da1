"""Seeded synthetic inputs for the int4 weight-only linear.

This module draws random numbers and nothing else: it holds none of the
quantization or matmul arithmetic, so both the CUDA path and the CPU oracle
can take their inputs from it.

The pages measure on real checkpoints (Llama-3-8B in the torchao README
overview and the torchao guide section 1.1/1.2; Gemma3-12b in the torchao
README "Inference" table).  Those weights are not available here; synthetic
tensors with Llama-3-8B linear shapes stand in for them:

* W ~ N(0, 0.02) drawn in fp32, optionally with 0.1 % outliers (each weight
  independently, Bernoulli p = 0.001, multiplied by 10), then rounded to bf16;
* X ~ N(0, 1) drawn in fp32 and rounded to bf16;
* every tensor has its own seed: ``1000 * config + 10 * layer + linear`` for
  weights, plus ``ACT_SEED_OFFSET`` for activations; config 1 uses seed 0.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

ACT_SEED_OFFSET = 1_000_000

# One transformer block of Llama-3-8B: (name, N = out features, K = in features).
LLAMA3_8B_LINEARS = (
    ("q", 4096, 4096),
    ("k", 1024, 4096),
    ("v", 1024, 4096),
    ("o", 4096, 4096),
    ("gate", 14336, 4096),
    ("up", 14336, 4096),
    ("down", 4096, 14336),
)
LLAMA3_8B_LAYERS = 32


@dataclass(frozen=True)
class LinearCase:
    """One linear of a workload: Y[M,N] = X[M,K] . dequant(W[N,K])^T."""
    name: str
    N: int
    K: int
    group_size: int
    M: int
    w_seed: int
    outliers: bool = False

    @property
    def x_seed(self) -> int:
        return self.w_seed + ACT_SEED_OFFSET


def weight_seed(config: int, layer: int = 0, linear: int = 0) -> int:
    if config == 1:
        return 0
    return 1000 * config + 10 * layer + linear


def gen_weight(N: int, K: int, seed: int, outliers: bool = False, device="cpu",
               std: float = 0.02) -> torch.Tensor:
    """bf16 [N,K]: N(0, std) in fp32, optional 0.1 % x10 outliers, rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn((N, K), generator=g, dtype=torch.float32, device=device)
    w.mul_(std)
    if outliers:
        mask = torch.rand((N, K), generator=g, dtype=torch.float32, device=device) < 1e-3
        w = torch.where(mask, w * 10.0, w)
    return w.to(torch.bfloat16)


def gen_activation(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """bf16 [M,K]: N(0, 1) in fp32 rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((M, K), generator=g, dtype=torch.float32, device=device).to(torch.bfloat16)


def config1():
    """Single 512x512 linear, g=32, M=1, seed 0 (torchao guide section 3.1 example shape)."""
    return [LinearCase("linear512", 512, 512, 32, 1, 0)]


def config2(layer: int = 0):
    """Llama-3-8B decode linears of one block, M=1, g=32, with 0.1 % x10 outliers."""
    return [LinearCase(n, N, K, 32, 1, weight_seed(2, layer, i), outliers=True)
            for i, (n, N, K) in enumerate(LLAMA3_8B_LINEARS)]


def config3():
    """Batched decode on the down / up projections, g=64, M in {2,4,8,16,32}."""
    out = []
    for i, (n, N, K) in enumerate((("down", 4096, 14336), ("up", 14336, 4096))):
        for M in (2, 4, 8, 16, 32):
            out.append(LinearCase(f"{n}_M{M}", N, K, 64, M, weight_seed(3, 0, i)))
    return out


def config4():
    """Prefill GEMMs, g=32, M in {2048, 8192}, (N,K) in {(14336,4096), (4096,14336)}."""
    out = []
    for i, (N, K) in enumerate(((14336, 4096), (4096, 14336))):
        for M in (2048, 8192):
            out.append(LinearCase(f"prefill_{N}x{K}_M{M}", N, K, 32, M, weight_seed(4, 0, i)))
    return out


def config5(M: int):
    """Full synthetic Llama-3-8B linear stack: 32 blocks x 7 linears, g=128, fresh X per linear."""
    return [LinearCase(f"L{l}.{n}", N, K, 128, M, weight_seed(5, l, i))
            for l in range(LLAMA3_8B_LAYERS) for i, (n, N, K) in enumerate(LLAMA3_8B_LINEARS)]


def config5_weight_count() -> int:
    return LLAMA3_8B_LAYERS * sum(N * K for _, N, K in LLAMA3_8B_LINEARS)
