"""Seeded synthetic inputs for the ConvRot INT8 linear, the SwiGLU MLP and the
small-M GEMV.

This module only draws random numbers: it holds none of the method's
arithmetic, and both the CUDA path and the CPU oracle are fed from it.  All
tensors are generated on the CPU with a seeded ``torch.Generator`` so the two
sides see bit-identical inputs.

Recipe (the shapes and distributions of the workloads on the source pages,
which used real Qwen-Image-2.1 / MiniMax-H3 checkpoints that are not available
here; synthetic tensors of the same shapes stand in for them):
  * activations: x ~ N(0, 1), rounded to bf16, with a fraction of outlier
    channels (the first round(frac * K) indices of a seeded permutation of K)
    multiplied by a factor before rounding;
  * weights: W ~ N(0, 1/K) in f32 (std 1/sqrt(K));
  * bias: b ~ N(0, 0.02^2) rounded to bf16 (std 0.02).
Each tensor gets its own derived seed, so generating one never shifts another.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = [
    "activation", "weight", "bias", "LinearCase", "MlpCase", "GemvCase",
    "LINEAR_TINY", "LINEAR_2048", "LINEAR_4096", "MLP_4096", "MLP_2048", "GEMV_CASES",
    "DIT_BLOCK", "bf16_bits",
]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def activation(M: int, K: int, seed: int, outlier_frac: float = 0.0,
               outlier_scale: float = 1.0) -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1) with round(outlier_frac * K) outlier channels x outlier_scale."""
    g = _gen(seed)
    x = torch.randn(M, K, generator=g, dtype=torch.float32)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        idx = torch.randperm(K, generator=g)[:n_out]
        x[:, idx] *= outlier_scale
    return x.to(torch.bfloat16)


def weight(N: int, K: int, seed: int) -> torch.Tensor:
    """f32 [N, K] ~ N(0, 1/K)."""
    return torch.randn(N, K, generator=_gen(seed), dtype=torch.float32) / math.sqrt(K)


def bias(N: int, seed: int, std: float = 0.02) -> torch.Tensor:
    """bf16 [N] ~ N(0, std^2)."""
    return (torch.randn(N, generator=_gen(seed), dtype=torch.float32) * std).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a CPU bf16 tensor as a numpy uint16 array."""
    import numpy as np
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass(frozen=True)
class LinearCase:
    """One ConvRot W8A8 linear: x bf16 [M, K] -> y bf16 [M, N]."""
    name: str
    M: int
    K: int
    N: int
    g: int
    seed: int
    outlier_frac: float
    outlier_scale: float
    with_bias: bool

    def x(self) -> torch.Tensor:
        return activation(self.M, self.K, 1000 * self.seed + 1, self.outlier_frac,
                          self.outlier_scale)

    def W(self) -> torch.Tensor:
        return weight(self.N, self.K, 1000 * self.seed + 2)

    def b(self):
        return bias(self.N, 1000 * self.seed + 3) if self.with_bias else None

    @property
    def ops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclass(frozen=True)
class MlpCase:
    """Fused SwiGLU MLP: x [M, H] -> packed [gate | up] [M, 2I] -> down [M, H]."""
    name: str
    M: int
    H: int
    I: int
    g: int
    seed: int
    outlier_frac: float
    outlier_scale: float
    with_bias: bool = False

    def x(self) -> torch.Tensor:
        return activation(self.M, self.H, 1000 * self.seed + 1, self.outlier_frac,
                          self.outlier_scale)

    def W_gate(self) -> torch.Tensor:
        return weight(self.I, self.H, 1000 * self.seed + 2)

    def W_up(self) -> torch.Tensor:
        return weight(self.I, self.H, 1000 * self.seed + 3)

    def W_down(self) -> torch.Tensor:
        return weight(self.H, self.I, 1000 * self.seed + 4)

    def b_gate_up(self):
        return bias(2 * self.I, 1000 * self.seed + 5) if self.with_bias else None

    def b_down(self):
        return bias(self.H, 1000 * self.seed + 6) if self.with_bias else None

    @property
    def ops(self) -> int:
        return 2 * self.M * (2 * self.I) * self.H + 2 * self.M * self.H * self.I


@dataclass(frozen=True)
class GemvCase:
    """Small-M decode GEMV: x bf16 [M <= 8, K] against an INT8 weight [N, K]."""
    name: str
    M: int
    K: int
    N: int
    g: int
    seed: int
    with_bias: bool = False

    def x(self) -> torch.Tensor:
        return activation(self.M, self.K, 1000 * self.seed + 1)

    def W(self) -> torch.Tensor:
        return weight(self.N, self.K, 1000 * self.seed + 2)

    def b(self):
        return bias(self.N, 1000 * self.seed + 3) if self.with_bias else None

    def algorithmic_bytes(self) -> int:
        # weight codes + f32 row scales + bf16 activation read + bf16 output write
        return self.N * self.K + 4 * self.N + 2 * self.M * self.K + 2 * self.M * self.N


# The workloads of the source pages, as synthetic stand-ins.
LINEAR_TINY = LinearCase("linear_tiny_64x256x128_g64", 64, 256, 128, 64, 0, 0.01, 20.0, True)
LINEAR_2048 = LinearCase("linear_2048x3072x1024_g128", 2048, 3072, 1024, 128, 1, 0.005, 30.0,
                         False)
LINEAR_4096 = LinearCase("linear_4096x4096x4096_g128", 4096, 4096, 4096, 128, 2, 0.005, 30.0,
                         False)
MLP_4096 = MlpCase("swiglu_mlp_4096_h3072_i12288_g128", 4096, 3072, 12288, 128, 3, 0.005, 30.0)
MLP_2048 = MlpCase("swiglu_mlp_2048_h3072_i1024_g128", 2048, 3072, 1024, 128, 4, 0.005, 30.0)
GEMV_CASES = tuple(
    GemvCase(f"gemv_m{M}_{N}x{K}_g128", M, K, N, 128, 5 + i)
    for i, (N, K) in enumerate(((12288, 4096), (4096, 12288), (18432, 3072)))
    for M in (1, 2, 4, 8)
)


@dataclass(frozen=True)
class DitBlock:
    """One DiT-shaped block of the 225-layer pass: qkv, attention-out, packed
    gate|up, swiglu down at M tokens, plus a modulation linear at M=1."""
    M: int = 4096
    hidden: int = 3072
    mlp: int = 12288
    g: int = 128
    blocks: int = 45
    linears: tuple = field(default=(("qkv", 3072, 9216), ("attn_out", 3072, 3072)))
    modulation: tuple = (3072, 18432)


DIT_BLOCK = DitBlock()
