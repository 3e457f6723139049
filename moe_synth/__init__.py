"""Seeded synthetic inputs for the MoE layer forward.

This module is the ONLY code shared by the CUDA path's tests/bench and the CPU
oracle. It draws random numbers and rounds them to the storage dtype; it holds
none of the layer's arithmetic (no gate, no softmax, no routing, no FFN).

Streams are independent per (seed, tensor id, block) so that any slice (one
expert's weights, one block of token rows) can be regenerated on its own:

    tensor id 0: x        [T, d]     blocks of 256 token rows, N(0, 1)
    tensor id 1: W_g      [d, N]     one block, N(0, 0.02^2), fp32
    tensor id 2: bias     [N]        Zipf-shaped expert bias (skewed workload only)
    tensor id 3: w_gate   [N, F, d]  one block per expert (W_1 of the GELU FFN)
    tensor id 4: w_up     [N, F, d]  one block per expert (SwiGLU only)
    tensor id 5: w_down   [N, d, F]  one block per expert (W_2 of the GELU FFN)

Weights are stored [out, in] (K-major rows), the layout the kernels and the
oracle both index. bf16 values are produced from fp32 draws by round to
nearest even and are returned as raw uint16 bit patterns (numpy has no bf16).
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

X_BLOCK_ROWS = 256
TID_X, TID_WG, TID_BIAS, TID_WGATE, TID_WUP, TID_WDOWN = 0, 1, 2, 3, 4, 5


@dataclass(frozen=True)
class Workload:
    """Shape and recipe of one MoE layer forward workload."""
    name: str
    T: int                # tokens (batch x seq flattened)
    d: int                # model dim
    N: int                # experts
    k: int                # experts per token
    F: int                # expert hidden dim (d_ff)
    act: str              # "swiglu" | "gelu_tanh"
    dtype: str            # "f32" | "bf16"  (activations and expert weights; gate is fp32)
    seed: int
    zipf_s: Optional[float] = None   # per-expert gate bias giving Zipf(s) expected load
    w_std: float = 0.02
    x_std: float = 1.0

    @property
    def A(self) -> int:
        return self.T * self.k

    @property
    def esize(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: a tiny fp32 case, a Mixtral-like prefill, the pages'
# worked example (4 x 2048 tokens, 64 experts, 4096 -> 16384 -> 4096, top-2),
# a decode-shaped batch and a Zipf-skewed load-imbalance case.
WORKLOADS = {
    "tiny-f32": Workload("tiny-f32", T=64, d=128, N=8, k=2, F=256, act="swiglu", dtype="f32", seed=1),
    "prefill-n8-f14336": Workload("prefill-n8-f14336", T=4096, d=4096, N=8, k=2, F=14336,
                                  act="swiglu", dtype="bf16", seed=2),
    "worked-example-n64-f16384-gelu": Workload("worked-example-n64-f16384-gelu", T=8192, d=4096, N=64,
                                               k=2, F=16384, act="gelu_tanh", dtype="bf16", seed=3),
    "decode-t32-n64-k8": Workload("decode-t32-n64-k8", T=32, d=3584, N=64, k=8, F=2560,
                                  act="swiglu", dtype="bf16", seed=4),
    "zipf-skew-n128-k8": Workload("zipf-skew-n128-k8", T=16384, d=2048, N=128, k=8, F=768,
                                  act="swiglu", dtype="bf16", seed=5, zipf_s=1.2),
    # profiling slice: the worked example's per-expert shape (~256 rows per expert,
    # 4096 -> 16384 -> 4096 GELU) with 8 of its 64 experts, 2.1 GB of weights
    "worked-example-slice-n8": Workload("worked-example-slice-n8", T=1024, d=4096, N=8, k=2, F=16384,
                                        act="gelu_tanh", dtype="bf16", seed=6),
    # profiling case of the grouping and the combine: the worked example's tokens, gate and routing
    # (same seed, T, d, N, k) with 128-wide experts, so x_perm / y_perm (134 MB) exceed L2 while the
    # weights take 0.2 GB
    "worked-example-f128": Workload("worked-example-f128", T=8192, d=4096, N=64, k=2, F=128,
                                    act="gelu_tanh", dtype="bf16", seed=3),
    # profiling case of the decode-shaped grouped GEMM: the decode batch's shapes with 16 experts
    # (0.88 GB of weights instead of 3.5 GB)
    "decode-slice-n16": Workload("decode-slice-n16", T=32, d=3584, N=16, k=8, F=2560, act="swiglu",
                                 dtype="bf16", seed=4),
    # profiling case of the decode batch's routing, grouping and combine: its tokens, gate and
    # routing (same seed, T, d, N, k) with 128-wide experts (0.18 GB of weights instead of 3.5 GB)
    "decode-f128": Workload("decode-f128", T=32, d=3584, N=64, k=8, F=128, act="swiglu", dtype="bf16",
                            seed=4),
}


def _rng(seed: int, tid: int, block: int) -> np.random.Generator:
    return np.random.default_rng([seed, tid, block])


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_f32(seed, tid, block, shape, std) -> np.ndarray:
    v = _rng(seed, tid, block).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    return v


def _store(v32: np.ndarray, dtype: str) -> np.ndarray:
    return v32 if dtype == "f32" else f32_to_bf16_bits(v32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Widen a stored tensor (fp32 array or bf16 bits) to fp64 exactly."""
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


def x_rows(w: Workload, t0: int, t1: int) -> np.ndarray:
    """Token rows [t0, t1) of x in the storage dtype (fp32 array or bf16 bits)."""
    out = np.empty((t1 - t0, w.d), dtype=np.float32 if w.dtype == "f32" else np.uint16)
    b0, b1 = t0 // X_BLOCK_ROWS, (t1 - 1) // X_BLOCK_ROWS
    for b in range(b0, b1 + 1):
        r0 = b * X_BLOCK_ROWS
        nrows = min(X_BLOCK_ROWS, w.T - r0)
        blk = _store(_normal_f32(w.seed, TID_X, b, (nrows, w.d), w.x_std), w.dtype)
        s0, s1 = max(t0, r0), min(t1, r0 + nrows)
        out[s0 - t0:s1 - t0] = blk[s0 - r0:s1 - r0]
    return out


def x_all(w: Workload) -> np.ndarray:
    return x_rows(w, 0, w.T)


def gate_weight(w: Workload) -> np.ndarray:
    """W_g [d, N] fp32 (the gate is kept in fp32 for every workload)."""
    return _normal_f32(w.seed, TID_WG, 0, (w.d, w.N), w.w_std)


def gate_bias(w: Workload) -> Optional[np.ndarray]:
    """Per-expert gate bias [N] fp32, or None.

    For zipf_s = s: p_r proportional to r^-s over ranks r = 1..N, ranks dealt to
    experts by a seeded permutation pi, and b_e = ln p_{pi(e)}. Adding b to the
    logits makes the expected selection frequency fall off like Zipf(s); the
    per-expert load cannot exceed T, so the realised histogram is flatter at the
    very top than the nominal Zipf shares.
    """
    if w.zipf_s is None:
        return None
    r = np.arange(1, w.N + 1, dtype=np.float64)
    p = r ** (-w.zipf_s)
    p /= p.sum()
    pi = _rng(w.seed, TID_BIAS, 0).permutation(w.N)
    return np.log(p[pi]).astype(np.float32)


def expert_weights(w: Workload, e: int):
    """(w_gate [F,d], w_up [F,d] or None, w_down [d,F]) of expert e, storage dtype."""
    wg = _store(_normal_f32(w.seed, TID_WGATE, e, (w.F, w.d), w.w_std), w.dtype)
    wu = _store(_normal_f32(w.seed, TID_WUP, e, (w.F, w.d), w.w_std), w.dtype) if w.act == "swiglu" else None
    wd = _store(_normal_f32(w.seed, TID_WDOWN, e, (w.d, w.F), w.w_std), w.dtype)
    return wg, wu, wd


def _expert_job(args):
    w, e = args
    return e, expert_weights(w, e)


def iter_expert_weights(w: Workload, experts=None, workers: Optional[int] = None):
    """Yield (e, (w_gate, w_up, w_down)) for the given experts, generated in a
    spawn-context process pool when the workload is large. Results arrive in
    completion order; each expert's values do not depend on the order."""
    experts = list(range(w.N)) if experts is None else list(experts)
    big = w.F * w.d * len(experts) > 64 * 1024 * 1024
    if workers is None:
        workers = min(len(os.sched_getaffinity(0)), 16) if big else 1
    if workers <= 1 or len(experts) <= 1:
        for e in experts:
            yield e, expert_weights(w, e)
        return
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        for e, ws in pool.imap_unordered(_expert_job, [(w, e) for e in experts], chunksize=1):
            yield e, ws


def all_expert_weights(w: Workload, workers: Optional[int] = None):
    """Stacked (w_gate [N,F,d], w_up [N,F,d] or None, w_down [N,d,F])."""
    dt = np.float32 if w.dtype == "f32" else np.uint16
    WG = np.empty((w.N, w.F, w.d), dtype=dt)
    WU = np.empty((w.N, w.F, w.d), dtype=dt) if w.act == "swiglu" else None
    WD = np.empty((w.N, w.d, w.F), dtype=dt)
    for e, (a, b, c) in iter_expert_weights(w, workers=workers):
        WG[e] = a
        if WU is not None:
            WU[e] = b
        WD[e] = c
    return WG, WU, WD
