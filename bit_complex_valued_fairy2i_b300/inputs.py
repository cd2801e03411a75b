"""Seeded synthetic inputs shaped like the pages' workload (LLaMA-2-7B linears).

This module holds no arithmetic of the method: it only draws random weights
and activations.  Both the oracle-based tests and the CUDA path take their
inputs from here.

Recipe:
  * weights  R ~ N(0, 0.02^2) float32, shape [2n, 2m] = [out, in] like a
    PyTorch Linear weight; seed = 20251203 + 1000*config + projection index.
  * activations x ~ N(0, 1) rounded to bfloat16, shape [M, 2m] (the model's
    real activation row, read as [Re x | Im x]); seed = weight seed + 500.
    With ``outliers`` each element is independently multiplied by 10 with
    probability 0.01 (mask drawn from the same generator after the values).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

BASE_SEED = 20251203
WEIGHT_STD = 0.02

# LLaMA-2-7B linear projections of one decoder block: (name, out, in).
LLAMA2_7B_BLOCK = (
    ("q_proj", 4096, 4096),
    ("k_proj", 4096, 4096),
    ("v_proj", 4096, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 11008, 4096),
    ("up_proj", 11008, 4096),
    ("down_proj", 4096, 11008),
)
LLAMA2_7B_BLOCKS = 32


@dataclass(frozen=True)
class Workload:
    name: str
    projections: tuple          # (name, out=2n, in=2m) per projection
    T: int
    M: tuple                    # token counts
    outliers: bool = False
    blocks: int = 1


WORKLOADS = {
    1: Workload("single layer 512x512, T=2, M=1", (("layer", 512, 512),), 2, (1,)),
    2: Workload("llama2-7b block decode, 7 projections, T=2, M=1", LLAMA2_7B_BLOCK, 2, (1,)),
    3: Workload("llama2-7b block batched decode sweep, T=2", LLAMA2_7B_BLOCK, 2,
                (1, 2, 4, 8, 16, 32, 64)),
    4: Workload("llama2-7b block prefill, M=2048, T=2, 1% outliers x10", LLAMA2_7B_BLOCK, 2,
                (2048,), outliers=True),
    5: Workload("llama2-7b 32-block linear stack, 224 projections, T in {1,2,3}, M=1",
                LLAMA2_7B_BLOCK, 2, (1,), blocks=LLAMA2_7B_BLOCKS),
}


def weight_seed(config: int, proj_index: int) -> int:
    return BASE_SEED + 1000 * config + proj_index


def weight_R(config: int, proj_index: int, out_features: int, in_features: int,
             device: str | torch.device = "cpu") -> torch.Tensor:
    """R ~ N(0, 0.02^2), float32 [out, in]."""
    g = torch.Generator(device=device)
    g.manual_seed(weight_seed(config, proj_index))
    R = torch.randn((out_features, in_features), generator=g, device=device, dtype=torch.float32)
    return R.mul_(WEIGHT_STD)


def activations(config: int, proj_index: int, M: int, in_features: int,
                outliers: bool = False, device: str | torch.device = "cpu") -> torch.Tensor:
    """x ~ N(0, 1) as bfloat16 [M, in]; optional 1 % outliers scaled by 10."""
    g = torch.Generator(device=device)
    g.manual_seed(weight_seed(config, proj_index) + 500)
    x = torch.randn((M, in_features), generator=g, device=device, dtype=torch.float32)
    if outliers:
        mask = torch.rand((M, in_features), generator=g, device=device) < 0.01
        x = torch.where(mask, x * 10.0, x)
    return x.to(torch.bfloat16)


def bf16_bits(x: torch.Tensor):
    """bfloat16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
