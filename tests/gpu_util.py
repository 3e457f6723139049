"""Helpers of the GPU parity tests: move seeded inputs to the device, run the
C-ABI calls, and compare with the CPU oracle under the stated bars:

  - top-k indices, counts, offsets, perm, inv_perm, x_perm: bit-exact on
    every token (the oracle takes the top-k decision on fp32 logits, the
    precision the pages fix for the gate);
  - bf16 outputs: max|out - ref| <= 2e-2 * max|ref|;
  - fp32 outputs: max|out - ref| <= 1e-4 * max|ref|;
  - top-k weights: 1e-5 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B

TOL_BF16 = 2e-2
TOL_F32 = 1e-4
TOL_W = 1e-5


def tol(dtype: str) -> float:
    return TOL_BF16 if dtype == "bf16" else TOL_F32


def dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays are bf16 bit patterns."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    m = float(np.max(np.abs(ref))) if ref.size else 0.0
    if m == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / m)


def check_route(gpu_idx: np.ndarray, gpu_w: np.ndarray, orc: dict) -> int:
    """Top-k indices bit-exact on every token against the oracle's fp32-gate
    decision; renormalised weights within 1e-5. Returns how many tokens the
    exact-logit certificate calls fragile (for reporting only)."""
    np.testing.assert_array_equal(gpu_idx, orc["topk_idx"])
    np.testing.assert_allclose(gpu_w, orc["topk_w"], rtol=0, atol=TOL_W)
    np.testing.assert_allclose(gpu_w.sum(1), 1.0, atol=1e-5)
    return int(np.sum(orc["cert"] <= 0))


def new(shape, dtype, fill=None):
    td = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32}[dtype]
    t = torch.empty(shape, dtype=td, device="cuda")
    if fill is not None:
        t.fill_(fill)
    return t


class Inputs:
    """A workload's seeded inputs on the device (and its small pieces on host)."""

    def __init__(self, w: S.Workload, host_weights: bool = True, on_expert=None):
        """on_expert(e, (w_gate, w_up, w_down)), if given, is called with each
        expert's host weights as they are uploaded (one pass over the weights
        serves the device copy and the oracle)."""
        self.w = w
        self.x_h = S.x_all(w)
        self.wg_h = S.gate_weight(w)
        self.bias_h = S.gate_bias(w)
        self.x = dev(self.x_h)
        self.wg = dev(self.wg_h)
        self.bias = dev(self.bias_h) if self.bias_h is not None else None
        td = B.TORCH_DTYPE[w.dtype]
        self.w_gate = torch.empty((w.N, w.F, w.d), dtype=td, device="cuda")
        self.w_up = torch.empty((w.N, w.F, w.d), dtype=td, device="cuda") if w.act == "swiglu" else None
        self.w_down = torch.empty((w.N, w.d, w.F), dtype=td, device="cuda")
        self.host = {} if host_weights else None
        for e, (a, b, c) in S.iter_expert_weights(w):
            self.w_gate[e].copy_(dev(a))
            if self.w_up is not None:
                self.w_up[e].copy_(dev(b))
            self.w_down[e].copy_(dev(c))
            if self.host is not None:
                self.host[e] = (a, b, c)
            if on_expert is not None:
                on_expert(e, (a, b, c))
        torch.cuda.synchronize()

    def expert(self, e):
        if self.host is not None:
            return self.host[e]
        return S.expert_weights(self.w, e)

    @property
    def shape(self):
        w = self.w
        return B.shape(w.T, w.d, w.N, w.k, w.F, w.act, w.dtype)


def run_forward(inp: Inputs, return_routing=True):
    w = inp.w
    s = inp.shape
    out = new((w.T, w.d), w.dtype)
    idx = new((w.T, w.k), "i32")
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    cnt = new((w.N,), "i32")
    ws = B.workspace(B.workspace_size(s))
    B.forward(s, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws,
              topk_idx=idx, topk_w=tw, counts=cnt)
    assert B.get_error() == B.MOE_OK
    return out, idx, tw, cnt


def oracle_outputs_for_tokens(inp: Inputs, tokens, topk_idx, topk_w):
    """fp64 layer output for the listed tokens, given their routing: each
    selected expert's FFN from the oracle, then the oracle's combine."""
    w = inp.w
    tokens = np.asarray(tokens, dtype=np.int64)
    by_e = {}
    for q, t in enumerate(tokens):
        for j in range(w.k):
            by_e.setdefault(int(topk_idx[t, j]), []).append((q, j))
    y = np.zeros((len(tokens) * w.k, w.d))
    for e, lst in by_e.items():
        a, b, c = inp.expert(e)
        rows = inp.x_h[[int(tokens[q]) for q, _ in lst]]
        ye = oracle.expert_rows(rows, a, b, c, w.act)
        for r, (q, j) in enumerate(lst):
            y[q * w.k + j] = ye[r]
    inv_local = np.arange(len(tokens) * w.k, dtype=np.int32)
    return oracle.combine(y, inv_local, np.asarray(topk_w)[tokens])
