"""Seeded synthetic inputs (bf16) shared by the tests, the benchmark and the
smoke check.  This module holds none of the FP8 method's arithmetic: it only
draws random tensors and rounds them to bf16.  The oracle and the CUDA path
receive the same bytes.

Workload shapes are those of 8B-class and 32B-class dense decoders (the
layer shapes the Jet-RL summaries' models have; no weights or datasets are
used):
  8B : hidden 4096, intermediate 14336, QKV out 6144 (32 heads, 8 KV heads)
  32B: hidden 5120, intermediate 27648, QKV out 7168
Distributions (all seeded, one sub-seed per tensor):
  X  ~ N(0, 1), optionally with round(1% of K) input channels (a seeded
       permutation) scaled by a factor (x20 for the 8B prefill / training
       shapes, x100 with Student-t(3) values for the 32B shapes);
  W  ~ N(0, 0.02);  dY ~ N(0, 1e-2) (8B) or N(0, 1e-3) (32B).
"""
from __future__ import annotations

import torch

PROJ_8B = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (28672, 4096), "down": (4096, 14336)}
PROJ_32B = {"qkv": (7168, 5120), "o": (5120, 5120), "gate_up": (55296, 5120), "down": (5120, 27648)}

TENSOR_IDS = {"x": 1, "w": 2, "dy": 3, "perm": 4, "chi": 5}


def _gen(seed: int, tensor: str, index: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + TENSOR_IDS[tensor] * 10_007 + index) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def normal_bf16(shape, sigma: float, seed: int, tensor: str, index: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, tensor, index, device)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * sigma).to(torch.bfloat16)


def student_t3_bf16(shape, seed: int, tensor: str, index: int = 0, device="cpu") -> torch.Tensor:
    """Student-t with 3 degrees of freedom: N / sqrt(chi2_3 / 3)."""
    g = _gen(seed, tensor, index, device)
    z = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    gc = _gen(seed, "chi", index, device)
    chi = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        chi += torch.randn(*shape, generator=gc, device=device, dtype=torch.float32) ** 2
    return (z / torch.sqrt(chi / 3.0)).to(torch.bfloat16)


def outlier_channels(K: int, seed: int, index: int = 0, device="cpu") -> torch.Tensor:
    """round(1% of K) channel indices from a seeded permutation."""
    g = _gen(seed, "perm", index, torch.device("cpu"))
    n = int(round(0.01 * K))
    return torch.randperm(K, generator=g)[:n].to(device)


def activation(M: int, K: int, seed: int, index: int = 0, device="cpu", outlier_scale: float = 0.0,
               student_t: bool = False) -> torch.Tensor:
    """X [M, K] bf16: N(0,1) or Student-t(3), optionally with 1% outlier channels
    scaled by ``outlier_scale`` before the bf16 rounding."""
    if student_t:
        g = _gen(seed, "x", index, device)
        z = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
        gc = _gen(seed, "chi", index, device)
        chi = torch.zeros(M, K, device=device, dtype=torch.float32)
        for _ in range(3):
            chi += torch.randn(M, K, generator=gc, device=device, dtype=torch.float32) ** 2
        x = z / torch.sqrt(chi / 3.0)
        del z, chi
    else:
        g = _gen(seed, "x", index, device)
        x = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    if outlier_scale:
        x[:, outlier_channels(K, seed, index, device)] *= outlier_scale
    return x.to(torch.bfloat16)


def weight(N: int, K: int, seed: int, index: int = 0, device="cpu") -> torch.Tensor:
    return normal_bf16((N, K), 0.02, seed, "w", index, device)


def grad_output(M: int, N: int, seed: int, index: int = 0, device="cpu", sigma: float = 1e-2) -> torch.Tensor:
    return normal_bf16((M, N), sigma, seed, "dy", index, device)


def bf16_bits(t: torch.Tensor):
    """CPU uint16 numpy view of a bf16 tensor's bit patterns (for the oracle)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def np_f32_to_bf16_bits(v):
    """bf16 bit patterns (uint16 numpy) of fp32 values, rounded to nearest even
    by PyTorch's own conversion."""
    import numpy as np
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view("uint16")
