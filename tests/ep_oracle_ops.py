"""The steps of the expert-parallel forward computed by the CPU oracle, for
checking the orchestration in mixture_experts_layer_97_b300.ep on hosts
without a GPU (host tensors; rows travel as raw bits, y rows in fp64).
Test infrastructure only."""
from __future__ import annotations

import numpy as np
import torch

import moe_synth as S
import oracle


def _t(a: np.ndarray) -> torch.Tensor:
    """numpy -> host tensor; bf16 bit patterns (uint16) travel as int16."""
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a))


def _np(t: torch.Tensor, bf16: bool) -> np.ndarray:
    a = t.numpy()
    return a.view(np.uint16) if bf16 and a.dtype == np.int16 else a


class OracleOps:
    def __init__(self, w: S.Workload, rank: int, part):
        self.w = w
        self.wg, self.bias = S.gate_weight(w), S.gate_bias(w)
        self.experts = {e: S.expert_weights(w, e) for e in part.experts(rank)}
        self.e0 = part.experts(rank)[0]
        self.bf16 = w.dtype == "bf16"

    def route_and_group(self, x):
        w = self.w
        xa = _np(x, self.bf16)
        r = oracle.route(xa, self.wg, w.k, bias=self.bias)
        p = oracle.permute(r["topk_idx"], w.N)
        return dict(idx=r["topk_idx"], tw=r["topk_w"], counts=_t(p["counts"]), inv=p["inv_perm"],
                    x_perm=_t(xa[p["perm"]]))

    def regroup(self, G, E, recv_counts, recv_x):
        g = oracle.ep_regroup(recv_counts)
        src = torch.from_numpy(g["local_src"].astype(np.int64))
        return recv_x[src], _t(g["offsets_local"]), _t(g["local_src"])

    def ffn(self, x_local, offsets_local, E):
        xa = _np(x_local, self.bf16)
        off = offsets_local.numpy()
        y = np.zeros((xa.shape[0], self.w.d))
        for e in range(E):
            a, b = int(off[e]), int(off[e + 1])
            if b > a:
                y[a:b] = oracle.expert_rows(xa[a:b], *self.experts[self.e0 + e], self.w.act)
        return torch.from_numpy(y)

    def ungroup(self, local_src, y_local):
        y = torch.empty_like(y_local)
        y[local_src.long()] = y_local
        return y

    def combine(self, y_perm, inv, tw):
        return torch.from_numpy(oracle.combine(y_perm.numpy(), inv, tw))

    def host_ints(self, t):
        return t.numpy()

    def rows(self, n, like):
        return torch.empty((int(n),) + tuple(like.shape[1:]), dtype=like.dtype)

    def check(self):
        pass
