"""Seeded synthetic inputs shared by the oracle tests, the CUDA parity tests and
the benchmark.  This module holds random draws and shapes only: none of the
quantizer's or the GEMM's arithmetic.

Every tensor is drawn on the CPU with ``numpy.random.default_rng(seed)``
(PCG64) in float32 and then rounded to BF16 (round-to-nearest-even, by
torch's CPU cast) where the workload is BF16, so the oracle and the GPU see
identical bytes.  "N(0, s)" is a normal with standard deviation s;
"t(nu) * s" is a Student-t draw with nu degrees of freedom times s.
Outlier positions are seeded draws without replacement.

The workloads are the shapes of the pages' experiments (Llama 3 8B and
Llama 3.1 405B MLP fprop, a Wgrad pass, routed-expert weights); no model,
weight or dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def normal(shape, std, seed) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def student_t(shape, nu, scale, seed) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_t(nu, size=shape).astype(np.float32) * np.float32(scale)).astype(np.float32)


def with_entry_outliers(x: np.ndarray, fraction: float, factor: float, seed: int) -> np.ndarray:
    """Multiply round(fraction * x.size) uniformly chosen entries by ``factor``."""
    rng = np.random.default_rng(seed)
    n = int(fraction * x.size)
    idx = rng.choice(x.size, size=n, replace=False)
    y = x.copy().reshape(-1)
    y[idx] *= np.float32(factor)
    return y.reshape(x.shape)


def with_channel_outliers(x: np.ndarray, fraction: float, factor: float, seed: int) -> np.ndarray:
    """Multiply round(fraction * cols) uniformly chosen columns by ``factor``."""
    rng = np.random.default_rng(seed)
    n = max(1, int(fraction * x.shape[1]))
    cols = rng.choice(x.shape[1], size=n, replace=False)
    y = x.copy()
    y[:, cols] *= np.float32(factor)
    return y


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy -> BF16 CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def bf16_to_f32_numpy(t: torch.Tensor) -> np.ndarray:
    """Exact BF16 -> float32 values as numpy (for the oracle)."""
    return t.to(torch.float32).numpy()


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------
@dataclass
class Workload:
    name: str
    tensors: dict = field(default_factory=dict)   # name -> CPU torch tensor (bf16 or f32)
    notes: str = ""


def pr1(seed_a=0, seed_b=1) -> Workload:
    """256x256 FP32, N(0,1), 1% of entries (655) x50; two such tensors."""
    a = with_entry_outliers(normal((256, 256), 1.0, seed_a), 0.01, 50.0, seed_a + 1000)
    b = with_entry_outliers(normal((256, 256), 1.0, seed_b), 0.01, 50.0, seed_b + 1000)
    return Workload("pr1_256_f32", {"A": torch.from_numpy(a), "B": torch.from_numpy(b)},
                    "A seed 0, B seed 1; outlier positions seed+1000")


def llama8b_fprop(m=8192, n=14336, k=4096) -> Workload:
    """X m x k BF16 N(0,1) with 0.1% of channels x20; W n x k BF16 N(0,0.02)."""
    x = with_channel_outliers(normal((m, k), 1.0, 2), 0.001, 20.0, 1002)
    w = normal((n, k), 0.02, 3)
    return Workload(f"llama3_8b_mlp_fprop_{m}x{n}x{k}", {"X": to_bf16(x), "W": to_bf16(w)})


def wgrad(tokens=8192, n_out=14336, n_in=4096) -> Workload:
    """dY tokens x n_out BF16 1e-3 * t(4); X tokens x n_in BF16 as in the 8B fprop."""
    dy = student_t((tokens, n_out), 4, 1e-3, 4)
    x = with_channel_outliers(normal((tokens, n_in), 1.0, 2), 0.001, 20.0, 1002)
    return Workload(f"wgrad_{n_out}x{n_in}x{tokens}", {"dY": to_bf16(dy), "X": to_bf16(x)})


def llama405b_fprop(m=8192, n=53248, k=16384) -> Workload:
    """X m x k BF16 N(0,1); W n x k BF16 N(0,0.01)."""
    x = normal((m, k), 1.0, 5)
    w = normal((n, k), 0.01, 6)
    return Workload(f"llama31_405b_mlp_fprop_{m}x{n}x{k}", {"X": to_bf16(x), "W": to_bf16(w)})


def moe(experts=64, tokens=512, k=4096, n=1536) -> Workload:
    """W experts x k x n BF16 0.02 * t(3) ([K][N] per expert); X experts x tokens x k BF16 N(0,1)."""
    w = student_t((experts, k, n), 3, 0.02, 7)
    x = normal((experts, tokens, k), 1.0, 8)
    return Workload(f"moe_{experts}x{tokens}x{n}x{k}", {"W": to_bf16(w), "X": to_bf16(x)})
