"""Seeded synthetic inputs shaped like the workloads the Jet-RL summary evaluates.

This module only draws random numbers; it holds none of the quantization or GEMM
arithmetic, and both the CUDA path and the CPU oracle consume what it returns.

Recipe (the pages evaluate Llama3.1-8B, Qwen2.5-7B and Qwen3-8B-Base RL runs with 8k-16k
token rollouts, section "Experimental results"; only their linear-layer shapes are used):
  * values ~ N(0, std) drawn in float32 with ``torch.Generator(device).manual_seed(seed)``
    (standard deviation ``std``), then rounded to BF16 (nearest even);
  * activations carry outlier channels: round(frac * K) distinct column indices (along the
    reduction dimension K) drawn by ``torch.randperm`` from the same generator, multiplied
    by ``outlier_scale`` before the BF16 rounding;
  * each tensor of a workload takes its own seed: ``seed * 1000 + index``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import torch


def normal_bf16(shape, std: float, seed: int, device="cpu", outlier_channels: int = 0,
                outlier_scale: float = 1.0) -> torch.Tensor:
    """N(0, std) values rounded to BF16, with optional scaled outlier columns."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(0.0, std, generator=g)
    if outlier_channels > 0:
        idx = torch.randperm(shape[-1], generator=g, device=device)[:outlier_channels]
        x[..., idx] *= outlier_scale
    return x.to(torch.bfloat16)


def outlier_count(frac: float, K: int) -> int:
    return int(round(frac * K))


@dataclass(frozen=True)
class Linear:
    """One linear layer Y[M,N] = X[M,K] W[N,K]^T."""
    name: str
    N: int
    K: int


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    M: List[int]
    linears: Tuple[Linear, ...]
    act_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_channels: int = 0   # fixed count (overrides outlier_frac when > 0)
    outlier_scale: float = 1.0
    weight_std: float = 0.02
    grad_std: float = 1e-3
    notes: str = ""
    extra: Dict[str, float] = field(default_factory=dict)


# Workloads named by what they are (model-shaped linears and token counts).
SINGLE_LINEAR_256x512 = Workload(
    name="single linear fwd 256x512x512", seed=0, M=[256],
    linears=(Linear("linear", 512, 512),), outlier_channels=4, outlier_scale=20.0,
    weight_std=0.02)

LLAMA8B_MLP_M8192 = Workload(
    name="Llama-3.1-8B MLP, 8192 tokens", seed=1, M=[8192],
    linears=(Linear("gate_up", 28672, 4096), Linear("down", 4096, 14336)),
    outlier_frac=0.001, outlier_scale=30.0, weight_std=0.02,
    extra={"eps": 1e-5})

LLAMA8B_MLP_BWD_M8192 = Workload(
    name="Llama-3.1-8B MLP backward, 8192 tokens", seed=2, M=[8192],
    linears=(Linear("gate_up", 28672, 4096), Linear("down", 4096, 14336)),
    outlier_frac=0.001, outlier_scale=30.0, weight_std=0.02, grad_std=1e-3)

QWEN7B_DECODE = Workload(
    name="Qwen2.5-7B linears, decode M in {64,128,256}", seed=3, M=[64, 128, 256],
    linears=(Linear("qkv", 4608, 3584), Linear("o", 3584, 3584),
             Linear("gate_up", 37888, 3584), Linear("down", 3584, 18944)),
    weight_std=0.02)

QWEN32B_LAYER_M16384 = Workload(
    name="Qwen2.5-32B layer, 16384 tokens", seed=4, M=[16384],
    linears=(Linear("qkv", 7168, 5120), Linear("o", 5120, 5120),
             Linear("gate_up", 55296, 5120), Linear("down", 5120, 27648)),
    outlier_frac=0.001, outlier_scale=30.0, weight_std=0.015, grad_std=1e-3)

WORKLOADS = [SINGLE_LINEAR_256x512, LLAMA8B_MLP_M8192, LLAMA8B_MLP_BWD_M8192, QWEN7B_DECODE,
             QWEN32B_LAYER_M16384]


def activation(w: Workload, M: int, K: int, index: int, device="cpu") -> torch.Tensor:
    n_out = w.outlier_channels if w.outlier_channels > 0 else outlier_count(w.outlier_frac, K)
    return normal_bf16((M, K), w.act_std, w.seed * 1000 + index, device, n_out,
                       w.outlier_scale)


def weight(w: Workload, lin: Linear, index: int, device="cpu") -> torch.Tensor:
    return normal_bf16((lin.N, lin.K), w.weight_std, w.seed * 1000 + index, device)


def gradient(w: Workload, M: int, N: int, index: int, device="cpu") -> torch.Tensor:
    return normal_bf16((M, N), w.grad_std, w.seed * 1000 + index, device)
