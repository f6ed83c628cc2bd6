"""Seeded synthetic input generators shared by the tests, the smoke check and
the benchmark.

This module holds no arithmetic of the reductions themselves: it only draws
random tensors with the shapes and value distributions of the workloads
(uniform / normal fp32, uniform int32, bf16-rounded normal logits and
activations, split-K attention partials).  Both the CUDA path and the CPU
oracle are fed from the same tensors it returns.
"""
from __future__ import annotations

import math

import torch

BASE_SEED = 20261202


def seed_for(config_index: int, op_index: int = 0) -> int:
    """Seed of one (workload, op) pair: base + 16 * workload + op."""
    return BASE_SEED + 16 * int(config_index) + int(op_index)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def uniform_f32(rows: int, cols: int, seed: int, device="cpu",
                lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    """x ~ Uniform[lo, hi) fp32, shape [rows, cols]."""
    g = _gen(seed, device)
    x = torch.rand((rows, cols), generator=g, device=device, dtype=torch.float32)
    return x.mul_(hi - lo).add_(lo)


def normal_f32(rows: int, cols: int, seed: int, device="cpu",
               std: float = 1.0) -> torch.Tensor:
    """x ~ N(0, std^2) fp32, shape [rows, cols]."""
    g = _gen(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def uniform_i32(rows: int, cols: int, seed: int, device="cpu",
                lo: int = -(1 << 15), hi: int = (1 << 15)) -> torch.Tensor:
    """x ~ UniformInt[lo, hi] int32 (both ends included)."""
    g = _gen(seed, device)
    return torch.randint(lo, hi + 1, (rows, cols), generator=g, device=device,
                         dtype=torch.int32)


def normal_bf16(rows: int, cols: int, seed: int, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    """x = bf16_rn(std * N(0,1)), shape [rows, cols] (fp32 draw rounded to
    bf16 nearest-even)."""
    return normal_f32(rows, cols, seed, device, std).to(torch.bfloat16)


def layernorm_params(cols: int, seed: int, device="cpu"):
    """Layernorm affine parameters: gamma = 1 + 0.1 N(0,1), beta = 0.1 N(0,1),
    fp32 [cols] each."""
    g = _gen(seed, device)
    gamma = torch.randn(cols, generator=g, device=device, dtype=torch.float32).mul_(0.1).add_(1.0)
    beta = torch.randn(cols, generator=g, device=device, dtype=torch.float32).mul_(0.1)
    return gamma, beta


def combine_partials(P: int, rows: int, D: int, seed: int, device="cpu"):
    """Split-K attention partials: per (p, row) l ~ U[1, 64), m ~ 2 * N(0,1);
    O[p, row, :] = N(0,1) * l[p, row].  Returns (O [P,rows,D], m [P,rows],
    l [P,rows]) fp32 and scale_log2e = fp32(log2(e) / sqrt(D))."""
    g = _gen(seed, device)
    l = torch.rand((P, rows), generator=g, device=device, dtype=torch.float32)
    l.mul_(63.0).add_(1.0)
    m = torch.randn((P, rows), generator=g, device=device, dtype=torch.float32)
    m.mul_(2.0)
    O = torch.randn((P, rows, D), generator=g, device=device, dtype=torch.float32)
    O.mul_(l.unsqueeze(-1))
    return O, m, l, scale_log2e_for(D)


def scale_log2e_for(D: int) -> float:
    """log2(e) / sqrt(D) computed in fp64 and rounded to fp32 once."""
    v = math.log2(math.e) / math.sqrt(D)
    return float(torch.tensor(v, dtype=torch.float64).to(torch.float32).item())
