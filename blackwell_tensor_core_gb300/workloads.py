"""Seeded synthetic inputs for the GEMM workloads (shared by tests and bench).

This module draws random numbers and nothing else: it holds none of the
GEMM's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it without sharing any of the method.

Every tensor is generated in float32 on the CPU from ``torch.Generator``
seeded per workload (seed = 1000 + workload index), then rounded to the input
dtype with round-to-nearest-even (``Tensor.to``).  The same bit patterns feed
the GPU and the oracle.

Workloads (shapes and value distributions of the method's five cases):
  1  tile      M=N=256, K=512, integers uniform in {-2..2}, FP32 output
  2  square    M=N=K=4096, N(0,1)/sqrt(K), BF16 output
  3  large     M=N=K=8192, U[-1,1], BF16 output
  4  small_m   M=72, N=16384, K=7168, N(0,1)*0.02, BF16 output
  5  grouped   32 experts, 32768 routed rows (top-8 of 4096 tokens), per-expert
               counts from a seeded multinomial, K=N=4096, A ~ N(0,1),
               B_g ~ N(0, 0.02), BF16 output (FC1; with SwiGLU, B_g = [gate | up])
  6  fc2       the same expert buckets (counts drawn as in 5), K=2048 (the
               SwiGLU width), N=4096, A ~ N(0,1), B_g ~ N(0, 0.02), BF16 output

Every case takes ``dtype`` ("bf16" or "fp16"): the same draws rounded to the
other input type (the FP16 runs use FP16 output).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

OUT_BF16 = 0
OUT_FP32 = 1
OUT_FP16 = 2

_TORCH_IN = {"bf16": torch.bfloat16, "fp16": torch.float16}


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def bits(t: torch.Tensor) -> np.ndarray:
    """The 16-bit patterns of a CPU bf16/fp16 tensor as numpy uint16 (no copy)."""
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("expected a 16-bit floating tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def randint_matrix(rows: int, cols: int, lo: int, hi: int, g: torch.Generator, dtype: str = "bf16"):
    """Integers uniform in [lo, hi] (inclusive), stored as bf16/fp16."""
    return torch.randint(lo, hi + 1, (rows, cols), generator=g, dtype=torch.int32).to(_TORCH_IN[dtype])


def normal_matrix(rows: int, cols: int, std: float, g: torch.Generator, dtype: str = "bf16"):
    return (torch.randn((rows, cols), generator=g, dtype=torch.float32) * std).to(_TORCH_IN[dtype])


def uniform_matrix(rows: int, cols: int, lo: float, hi: float, g: torch.Generator, dtype: str = "bf16"):
    u = torch.rand((rows, cols), generator=g, dtype=torch.float32)
    return (u * (hi - lo) + lo).to(_TORCH_IN[dtype])


def expert_counts(tokens: int, topk: int, experts: int, g: torch.Generator) -> np.ndarray:
    """Per-expert row counts: tokens*topk draws from a uniform multinomial over
    the experts (with replacement), counted per expert.  Zero counts are legal."""
    draws = torch.multinomial(torch.ones(experts), tokens * topk, replacement=True, generator=g)
    return torch.bincount(draws, minlength=experts).numpy().astype(np.int64)


def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(len(counts) + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off


@dataclass
class Dense:
    name: str
    M: int
    N: int
    K: int
    A: torch.Tensor  # [M, K] CPU
    B: torch.Tensor  # [K, N] CPU
    out_dtype: int
    in_dtype: str = "bf16"

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclass
class Grouped:
    name: str
    N: int
    K: int
    A: torch.Tensor  # [total, K]
    Bs: list = field(default_factory=list)  # G x [K, N]
    offsets: np.ndarray = None  # int32 [G+1]
    in_dtype: str = "bf16"

    @property
    def G(self) -> int:
        return len(self.Bs)

    @property
    def total(self) -> int:
        return int(self.offsets[-1])

    @property
    def flops(self) -> int:
        return 2 * self.total * self.N * self.K


def _out_for(dtype: str) -> int:
    return OUT_FP16 if dtype == "fp16" else OUT_BF16


def tile_case(seed: int = 1001, dtype: str = "bf16") -> Dense:
    g = generator(seed)
    A = randint_matrix(256, 512, -2, 2, g, dtype)
    B = randint_matrix(512, 256, -2, 2, g, dtype)
    return Dense("tile_256x256x512_int", 256, 256, 512, A, B, OUT_FP32, dtype)


def square_case(seed: int = 1002, n: int = 4096, dtype: str = "bf16") -> Dense:
    g = generator(seed)
    A = normal_matrix(n, n, 1.0 / math.sqrt(n), g, dtype)
    B = normal_matrix(n, n, 1.0 / math.sqrt(n), g, dtype)
    return Dense("square_%d_%s" % (n, dtype), n, n, n, A, B, _out_for(dtype), dtype)


def large_case(seed: int = 1003, n: int = 8192, dtype: str = "bf16") -> Dense:
    g = generator(seed)
    A = uniform_matrix(n, n, -1.0, 1.0, g, dtype)
    B = uniform_matrix(n, n, -1.0, 1.0, g, dtype)
    return Dense("large_%d_%s" % (n, dtype), n, n, n, A, B, _out_for(dtype), dtype)


def small_m_case(seed: int = 1004, M: int = 72, N: int = 16384, K: int = 7168,
                 dtype: str = "bf16") -> Dense:
    g = generator(seed)
    A = normal_matrix(M, K, 0.02, g, dtype)
    B = normal_matrix(K, N, 0.02, g, dtype)
    return Dense("small_m_%dx%dx%d_%s" % (M, N, K, dtype), M, N, K, A, B, _out_for(dtype), dtype)


def grouped_case(seed: int = 1005, tokens: int = 4096, topk: int = 8, experts: int = 32,
                 N: int = 4096, K: int = 4096, dtype: str = "bf16") -> Grouped:
    g = generator(seed)
    counts = expert_counts(tokens, topk, experts, g)
    off = offsets_from_counts(counts)
    A = normal_matrix(int(off[-1]), K, 1.0, g, dtype)
    Bs = [normal_matrix(K, N, 0.02, g, dtype) for _ in range(experts)]
    return Grouped("grouped_fc1_%dx%d_E%d_%s" % (N, K, experts, dtype), N, K, A, Bs, off, dtype)


def grouped_fc2_case(seed: int = 1006, tokens: int = 4096, topk: int = 8, experts: int = 32,
                     N: int = 4096, K: int = 2048, dtype: str = "bf16") -> Grouped:
    """Expert FC2 (down projection) over the FC1 case's token buckets: the
    counts are drawn exactly as the FC1 case draws them (its seed, first draw),
    the activations and weights from this case's own seed."""
    counts = expert_counts(tokens, topk, experts, generator(1005))
    off = offsets_from_counts(counts)
    g = generator(seed)
    A = normal_matrix(int(off[-1]), K, 1.0, g, dtype)
    Bs = [normal_matrix(K, N, 0.02, g, dtype) for _ in range(experts)]
    return Grouped("grouped_fc2_%dx%d_E%d_%s" % (N, K, experts, dtype), N, K, A, Bs, off, dtype)


def case(index: int) -> Dense | Grouped:
    """The method workloads by index (1-based, as listed in the docstring)."""
    return {1: tile_case, 2: square_case, 3: large_case, 4: small_m_case, 5: grouped_case,
            6: grouped_fc2_case}[index]()
