"""Seeded synthetic inputs and the Qwen3 projection shapes.

This module holds no arithmetic of the method: it only draws random inputs of
the documented shapes, dtypes and value ranges, on the CPU, from a seeded
``torch.Generator``. Both the CUDA path and the CPU oracle consume what it
produces, so neither can influence the other's inputs.

Shapes follow the page "Qwen3 CPU Inference Critical Path" (section "Frozen
model contract", the model table: hidden 1,024 / 2,560, intermediate
3,072 / 9,728, 16/32 query heads and 8 KV heads of size 128, vocabulary
151,936, 28 / 36 layers; section "Exact kernel inventory", MatMulNBits row:
the projection shapes and block size 32).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Projection:
    name: str
    K: int  # input features
    N: int  # output features


def qwen3_projections(hidden: int, intermediate: int, q_heads: int,
                      kv_heads: int, head: int = 128) -> list[Projection]:
    """The seven per-layer projections of a dense Qwen3 decoder layer."""
    return [
        Projection("q", hidden, q_heads * head),
        Projection("k", hidden, kv_heads * head),
        Projection("v", hidden, kv_heads * head),
        Projection("o", q_heads * head, hidden),
        Projection("gate", hidden, intermediate),
        Projection("up", hidden, intermediate),
        Projection("down", intermediate, hidden),
    ]


VOCAB = 151936
QWEN3_0P6B = dict(layers=28, projections=qwen3_projections(1024, 3072, 16, 8),
                  lm_head=Projection("lm_head", 1024, VOCAB))
QWEN3_4B = dict(layers=36, projections=qwen3_projections(2560, 9728, 32, 8),
                lm_head=Projection("lm_head", 2560, VOCAB))


@dataclass
class Problem:
    """One MatMulNBits problem in the operator's input layout (CPU tensors)."""
    M: int
    N: int
    K: int
    block_size: int
    A: torch.Tensor                      # [M, K] float32 or bfloat16
    B: torch.Tensor                      # uint8 [N, nb, bs/2]
    scales: torch.Tensor                 # [N, nb], A's dtype
    zero_points: torch.Tensor | None     # uint8 [N, ceil(nb/2)] or None
    bias: torch.Tensor | None            # float32 [N] or None

    @property
    def n_blocks(self) -> int:
        return (self.K + self.block_size - 1) // self.block_size

    def algorithmic_bytes(self) -> int:
        """Bytes one call must move at least: packed B, scales, zero points,
        A, Y and bias, in their stored dtypes."""
        es = self.A.element_size()
        nb = self.n_blocks
        total = self.N * nb * (self.block_size // 2)
        total += self.N * nb * self.scales.element_size()
        if self.zero_points is not None:
            total += self.N * ((nb + 1) // 2)
        total += self.M * self.K * es + self.M * self.N * es
        if self.bias is not None:
            total += 4 * self.N
        return total

    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def make_problem(M: int, N: int, K: int, block_size: int = 32, *,
                 dtype: torch.dtype = torch.float32, zero_points: bool = False,
                 bias: bool = False, seed: int = 0,
                 scale_range: tuple[float, float] = (0.005, 0.02),
                 bias_std: float = 0.02) -> Problem:
    """Seeded synthetic problem: A ~ N(0,1); every byte of B uniform over
    0..255 (so both nibbles are uniform over 0..15); scales uniform over
    ``scale_range`` drawn in fp32 and then stored in A's dtype; zero-point
    bytes uniform over 0..255; bias ~ N(0, bias_std^2) in fp32."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    nb = (K + block_size - 1) // block_size
    A = torch.randn(M, K, generator=g, dtype=torch.float32).to(dtype)
    B = torch.randint(0, 256, (N, nb, block_size // 2), generator=g,
                      dtype=torch.uint8)
    lo, hi = scale_range
    scales = (torch.rand(N, nb, generator=g, dtype=torch.float32)
              * (hi - lo) + lo).to(dtype)
    zp = (torch.randint(0, 256, (N, (nb + 1) // 2), generator=g,
                        dtype=torch.uint8) if zero_points else None)
    b = (torch.randn(N, generator=g, dtype=torch.float32) * bias_std
         if bias else None)
    return Problem(M, N, K, block_size, A, B, scales, zp, b)


def decode_step_problems(model: dict, *, dtype: torch.dtype, block_size: int,
                         zero_points: bool, scale_range: tuple[float, float],
                         seed_base: int, layers: int | None = None,
                         lm_head: bool = True) -> list[tuple[str, Problem]]:
    """Every projection of one batch-1 decode step (M = 1), each with its own
    seeded weights and activation row. Seed = seed_base + running index."""
    out = []
    idx = 0
    n_layers = model["layers"] if layers is None else layers
    for layer in range(n_layers):
        for p in model["projections"]:
            out.append((f"L{layer}.{p.name}",
                        make_problem(1, p.N, p.K, block_size, dtype=dtype,
                                     zero_points=zero_points, seed=seed_base + idx,
                                     scale_range=scale_range)))
            idx += 1
    if lm_head:
        p = model["lm_head"]
        out.append((p.name, make_problem(1, p.N, p.K, block_size, dtype=dtype,
                                          zero_points=zero_points,
                                          seed=seed_base + idx,
                                          scale_range=scale_range)))
    return out
