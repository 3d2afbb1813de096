"""Seeded synthetic inputs and the named attention workloads.

This module only draws random numbers and names shapes; it holds none of the
attention arithmetic. It is the one module that both the CUDA path's tests /
benchmark and the fp64 oracle's callers use, so that both sides see the same
bf16 values.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws
Q, K, V, dO in that order as fp32 standard normals, Q and K are multiplied by
``qk_std``, and each tensor is rounded to bf16 (round-to-nearest-even). The
oracle consumes these exact bf16 values widened to fp64.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    m: int
    d: int
    causal: bool
    qk_std: float
    seed: int

    @property
    def heads(self) -> int:
        return self.B * self.H

    def flops_fwd(self) -> float:
        """4*B*H*n*m*d per forward, halved under causal masking."""
        f = 4.0 * self.B * self.H * self.n * self.m * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        """2.5 times the forward count."""
        return 2.5 * self.flops_fwd()

    def describe(self) -> str:
        c = "causal" if self.causal else "non-causal"
        return (f"B={self.B},H={self.H},n={self.n},m={self.m},d={self.d},{c},"
                f"Q,K~{self.qk_std:g}*N(0,1),V,dO~N(0,1),bf16,seed={self.seed}")


# The five workloads of the exact-attention study (seed 1000 + k for the k-th).
SINGLE_HEAD_128 = Workload("single_head_n128_d64", 1, 1, 128, 128, 64, False, 1.0, 1001)
SINGLE_HEAD_128_CAUSAL = Workload("single_head_n128_d64_causal", 1, 1, 128, 128, 64, True,
                                  1.0, 1001)
B4_H16_N1024_D64 = Workload("b4_h16_n1024_d64_causal", 4, 16, 1024, 1024, 64, True, 1.0, 1002)
LLAMA_B2_H32_N4096_D128 = Workload("llama_b2_h32_n4096_d128_causal", 2, 32, 4096, 4096, 128,
                                   True, 1.0, 1003)
LONG_B1_H16_N16384_D128 = Workload("long_b1_h16_n16384_d128_causal", 1, 16, 16384, 16384, 128,
                                   True, 1.0, 1004)
CROSS_B8_H8_N1000_M3000_D64 = Workload("cross_b8_h8_n1000_m3000_d64", 8, 8, 1000, 3000, 64,
                                       False, 3.0, 1005)

WORKLOADS = {w.name: w for w in (SINGLE_HEAD_128, SINGLE_HEAD_128_CAUSAL, B4_H16_N1024_D64,
                                 LLAMA_B2_H32_N4096_D128, LONG_B1_H16_N16384_D128,
                                 CROSS_B8_H8_N1000_M3000_D64)}


def attention_inputs(B: int, H: int, n: int, m: int, d: int, seed: int, qk_std: float = 1.0):
    """Q, dO: bf16 [B,H,n,d]; K, V: bf16 [B,H,m,d] on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    Q = torch.randn(B, H, n, d, generator=g, dtype=torch.float32)
    K = torch.randn(B, H, m, d, generator=g, dtype=torch.float32)
    V = torch.randn(B, H, m, d, generator=g, dtype=torch.float32)
    dO = torch.randn(B, H, n, d, generator=g, dtype=torch.float32)
    if qk_std != 1.0:
        Q.mul_(qk_std)
        K.mul_(qk_std)
    return (Q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16),
            dO.to(torch.bfloat16))


def workload_inputs(w: Workload):
    return attention_inputs(w.B, w.H, w.n, w.m, w.d, w.seed, w.qk_std)


def sample_indices(count: int, k: int, seed: int):
    """``k`` distinct indices in [0, count), sorted, from a seeded generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    k = min(k, count)
    return torch.randperm(count, generator=g)[:k].sort().values.tolist()


def score_rows(rows: int, cols: int, seed: int, std: float = 5.0) -> torch.Tensor:
    """fp32 [rows, cols] standard normals times `std` from a seeded CPU generator
    (the pages' online-softmax demo draws randn(10) * 5)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn(rows, cols, generator=g, dtype=torch.float32) * std
