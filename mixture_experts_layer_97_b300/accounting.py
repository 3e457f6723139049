"""FLOP and byte accounting for the MoE layer forward (host logic, no CUDA).

Counts are algorithmic: 2 FLOPs per multiply-add; bytes are what each step
must move at least once. The per-token-per-expert FLOP formula is the one of
"MoE混合专家模型计算原理与推理部署实战解析" section 3.4 (three d x d_ff projections
for SwiGLU); the two-matrix FFN of "MoE显存与计算开销四阶段手算指南" section 2 has two.
"""
from __future__ import annotations

from typing import Optional, Sequence


def n_proj(act: str) -> int:
    return 3 if act == "swiglu" else 2


def ffn_flops_per_assignment(d: int, F: int, act: str) -> float:
    return 2.0 * n_proj(act) * d * F


def ffn_flops(A: int, d: int, F: int, act: str) -> float:
    """Grouped expert FFN FLOPs for A token-expert assignments."""
    return A * ffn_flops_per_assignment(d, F, act)


def up_flops(A: int, d: int, F: int, act: str) -> float:
    """The first grouped GEMM (gate+up for SwiGLU, W_1 for GELU)."""
    return 2.0 * (n_proj(act) - 1) * A * d * F


def down_flops(A: int, d: int, F: int) -> float:
    return 2.0 * A * d * F


def gate_flops(T: int, d: int, N: int) -> float:
    return 2.0 * T * d * N


def layer_flops(T: int, d: int, N: int, k: int, F: int, act: str) -> float:
    return gate_flops(T, d, N) + ffn_flops(T * k, d, F, act)


def expert_weight_bytes(d: int, F: int, act: str, esize: int) -> int:
    return n_proj(act) * d * F * esize


def active_expert_weight_bytes(counts: Sequence[int], d: int, F: int, act: str, esize: int) -> int:
    """Weights every active expert must stream from HBM once."""
    return sum(1 for c in counts if c > 0) * expert_weight_bytes(d, F, act, esize)


def decode_forward_bytes(counts: Sequence[int], T: int, d: int, N: int, k: int, F: int,
                         act: str, esize: int) -> int:
    """Minimum HBM bytes of one forward when weights dominate: active experts'
    weights + x + W_g (fp32) + out + top-k outputs."""
    return (active_expert_weight_bytes(counts, d, F, act, esize)
            + T * d * esize * 2 + d * N * 4 + T * k * 8)


def permute_bytes(T: int, d: int, k: int, esize: int) -> int:
    """x read once, x_perm written for every assignment, indices."""
    A = T * k
    return T * d * esize + A * d * esize + A * 4 * 3 + T * k * 4


def combine_bytes(T: int, d: int, k: int, esize: int) -> int:
    """y_perm read for every assignment, out written, weights and indices."""
    A = T * k
    return A * d * esize + T * d * esize + A * 8


def route_bytes(T: int, d: int, N: int, k: int, esize: int) -> int:
    return T * d * esize + d * N * 4 + T * k * 8
