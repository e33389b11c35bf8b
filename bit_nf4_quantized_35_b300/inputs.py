"""Seeded synthetic inputs for the QLoRA NF4 linear-layer hot path.

This module is shared by the tests, the smoke check and the benchmark.  It
holds NO arithmetic of the method (no quantisation, no dequantisation, no
contraction): it only draws random tensors of the right shapes,
distributions and seeds, so that the CUDA path and the CPU oracle can be fed
identical inputs.

Recipe (every tensor drawn by torch's CPU generator in binary32, then
multiplied by its standard deviation in binary32, then rounded to nearest
even bf16 unless stated):
  - base weight W [N, K] ~ N(0, 0.02)          seed 0 (fp32 kept for the
                                                256x256 case)
  - activations x [M, K] ~ N(0, 1)              seed 1
  - LoRA A [r, K] ~ N(0, 0.01)                  seed 2
  - LoRA B [N, r] ~ N(0, 0.01)  (non-zero)      seed 3
  - upstream gradient dY [M, N] ~ N(0, 1)       seed 4
  - bulk quantisation matrix i [4096, 14336] ~ N(0, 0.02) with each entry
    independently replaced, with probability 0.001, by +-0.2 (10 sigma, fair
    sign); seed 1000 + i.
The shapes follow the workloads described on the pages: a single 256x256
layer, a 4096x4096 q_proj-shaped projection at 2048 tokens, a 4096->14336
gate_proj-shaped decode GEMV with 1, 4 or 16 tokens, the Llama-3-8B
projection set (q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096, down
4096x14336) at 4x2048 tokens, and 136 bulk 4096x14336 matrices.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SEED_W, SEED_X, SEED_A, SEED_B, SEED_DY = 0, 1, 2, 3, 4
SEED_BULK_BASE = 1000

STD_W, STD_X, STD_LORA, STD_DY = 0.02, 1.0, 0.01, 1.0
OUTLIER_P, OUTLIER_SIGMA = 0.001, 10.0


def _gen(seed: int, device: str = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, dtype=torch.bfloat16, device: str = "cpu") -> torch.Tensor:
    """N(0, std) drawn in binary32 with the given seed, then cast to ``dtype``."""
    g = _gen(seed, device)
    v = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    v.mul_(std)
    return v if dtype == torch.float32 else v.to(dtype)


def bulk_matrix(i: int, rows: int = 4096, cols: int = 14336, device: str = "cpu",
                dtype=torch.bfloat16) -> torch.Tensor:
    """Bulk-quantisation matrix number ``i``: N(0, 0.02) with 0.1 % +-10 sigma
    outliers (Bernoulli per entry, fair sign)."""
    g = _gen(SEED_BULK_BASE + i, device)
    v = torch.randn((rows, cols), generator=g, dtype=torch.float32, device=device)
    v.mul_(STD_W)
    u = torch.rand((rows, cols), generator=g, dtype=torch.float32, device=device)
    s = torch.rand((rows, cols), generator=g, dtype=torch.float32, device=device)
    out_val = torch.where(s < 0.5, -OUTLIER_SIGMA * STD_W, OUTLIER_SIGMA * STD_W)
    v = torch.where(u < OUTLIER_P, out_val, v)
    return v.to(dtype)


@dataclass(frozen=True)
class LinearShape:
    name: str
    N: int          # out features (rows of W)
    K: int          # in features (cols of W)
    M: int          # tokens
    r: int
    alpha: float
    w_dtype: torch.dtype = torch.bfloat16


def linear_inputs(shape: LinearShape, device: str = "cpu", with_dy: bool = True,
                  seed_offset: int = 0) -> dict:
    """W, x, A, B (and dY) for one QLoRA linear layer, seeded per the recipe."""
    so = seed_offset
    d = {
        "W": normal((shape.N, shape.K), STD_W, SEED_W + so, shape.w_dtype, device),
        "x": normal((shape.M, shape.K), STD_X, SEED_X + so, torch.bfloat16, device),
        "A": normal((shape.r, shape.K), STD_LORA, SEED_A + so, torch.bfloat16, device),
        "B": normal((shape.N, shape.r), STD_LORA, SEED_B + so, torch.bfloat16, device),
    }
    if with_dy:
        d["dY"] = normal((shape.M, shape.N), STD_DY, SEED_DY + so, torch.bfloat16, device)
    return d


# Workloads ---------------------------------------------------------------
SINGLE_256 = LinearShape("single_256x256_r8", N=256, K=256, M=4, r=8, alpha=16.0,
                         w_dtype=torch.float32)
QPROJ_2048 = LinearShape("q_proj_4096x4096_M2048_r16", N=4096, K=4096, M=2048, r=16,
                         alpha=32.0)


def gate_decode(M: int) -> LinearShape:
    return LinearShape(f"gate_proj_14336x4096_M{M}_r16", N=14336, K=4096, M=M, r=16,
                       alpha=32.0)


LLAMA3_8B_PROJ = {
    # name: (out N, in K)
    "q_proj": (4096, 4096),
    "k_proj": (1024, 4096),
    "v_proj": (1024, 4096),
    "o_proj": (4096, 4096),
    "gate_proj": (14336, 4096),
    "up_proj": (14336, 4096),
    "down_proj": (4096, 14336),
}


def llama3_layer_set(M: int = 8192) -> list[LinearShape]:
    return [LinearShape(f"{name}_M{M}", N=n, K=k, M=M, r=16, alpha=32.0)
            for name, (n, k) in LLAMA3_8B_PROJ.items()]


BULK_MATRICES = 136          # 136 x 4096 x 14336 = 7.986e9 weights
BULK_ROWS, BULK_COLS = 4096, 14336
