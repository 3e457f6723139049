"""Expert-parallel MoE layer forward over the ranks of a torch.distributed group.

"MoE混合专家模型计算原理与推理部署实战解析" section 3.3: when the experts do not
fit one GPU they are split over GPUs by expert id (8 experts over 4 cards, 2
each), every card routes its own tokens, and an all-to-all carries each token
row to the card that holds its expert (traffic proportional to tokens x hidden
size); section 6.3 calls this expert parallelism (EP). Reading: rank g of G
holds the contiguous experts [g E, (g + 1) E), E = N / G.

One forward on every rank, with its own tokens x [T, d] and its own experts'
weights:

  1. route and group its tokens (moe_route, moe_permute): x_perm is ordered by
     expert, hence by destination rank;
  2. all-to-all of the per-expert row counts (G x E integers per rank);
  3. all-to-all of the x_perm rows (split by destination rank);
  4. moe_ep_regroup: the received rows, ordered (source, local expert), grouped
     by local expert;
  5. moe_grouped_ffn over the local experts;
  6. moe_ep_ungroup back to the received order, and the reverse all-to-all,
     which returns every row to its source as that source's y_perm;
  7. moe_combine on the source, unchanged.

All compute runs in the library's kernels (``CudaOps``); this module only
orders the calls and moves rows with torch.distributed (NCCL on device
tensors; a CPU-only backend such as gloo gets the rows through host
memory). The ops object is a parameter so that the same orchestration can be
checked on a host without a GPU against another implementation of the steps.
"""
from __future__ import annotations

from dataclasses import dataclass
import numpy as np
import torch

from . import binding as B


@dataclass(frozen=True)
class Partition:
    """Experts split over G ranks in contiguous id ranges of E = N / G."""
    N: int
    G: int

    def __post_init__(self):
        if self.G < 1 or self.N % self.G != 0:
            raise ValueError(f"{self.N} experts do not split evenly over {self.G} ranks")

    @property
    def E(self) -> int:
        return self.N // self.G

    def experts(self, g: int) -> range:
        return range(g * self.E, (g + 1) * self.E)

    def send_counts(self, counts: np.ndarray) -> np.ndarray:
        """Rows this rank sends to each rank: its expert counts summed per range."""
        return np.asarray(counts, dtype=np.int64).reshape(self.G, self.E).sum(axis=1)


class CudaOps:
    """The forward's local steps through the C ABI (device tensors).

    w_gate / w_up / w_down hold this rank's E experts only ([E, F, d] /
    [E, F, d] or None / [E, d, F])."""

    def __init__(self, s: B.MoeShape, dtype: str, w_g, bias, w_gate, w_up, w_down, stream=None):
        self.s = s
        self.dtype = dtype
        self.w_g, self.bias = w_g, bias
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.stream = stream
        self.device = w_gate.device
        self.tdtype = B.TORCH_DTYPE[dtype]

    def _i32(self, n):
        return torch.empty(max(int(n), 0), dtype=torch.int32, device=self.device)

    def route_and_group(self, x):
        s = self.s
        T, k, N, d = int(s.T), int(s.k), int(s.N), int(s.d)
        idx = torch.empty((T, k), dtype=torch.int32, device=self.device)
        tw = torch.empty((T, k), dtype=torch.float32, device=self.device)
        B.route(s, x, self.w_g, self.bias, idx, tw, stream=self.stream)
        counts, offsets = self._i32(N), self._i32(N + 1)
        perm, inv = self._i32(T * k), self._i32(T * k)
        xp = torch.empty((T * k, d), dtype=self.tdtype, device=self.device)
        B.permute(s, idx, x, counts, offsets, perm, inv, xp, B.workspace(B.permute_workspace_size(s)),
                  stream=self.stream)
        return dict(idx=idx, tw=tw, counts=counts, inv=inv, x_perm=xp)

    def regroup(self, G, E, recv_counts: np.ndarray, recv_x):
        rows = int(recv_x.shape[0])
        rc = torch.from_numpy(np.ascontiguousarray(recv_counts, dtype=np.int32)).to(self.device)
        x_local = torch.empty_like(recv_x)
        offsets_local, local_src = self._i32(E + 1), self._i32(rows)
        B.ep_regroup(G, E, rc, recv_x, x_local, offsets_local, local_src, self.dtype, stream=self.stream)
        return x_local, offsets_local, local_src

    def ffn(self, x_local, offsets_local, E):
        s = self.s
        rows = int(x_local.shape[0])
        sl = B.shape(rows, int(s.d), E, 1, int(s.d_ff), "swiglu" if s.act == B.MOE_SWIGLU else "gelu_tanh",
                     self.dtype)
        y = torch.empty_like(x_local)
        if rows:
            B.grouped_ffn(sl, x_local, offsets_local, self.w_gate, self.w_up, self.w_down, y,
                          B.workspace(B.grouped_ffn_workspace_size(sl)), stream=self.stream)
        return y

    def ungroup(self, local_src, y_local):
        y_recv = torch.empty_like(y_local)
        B.ep_ungroup(local_src, y_local, y_recv, self.dtype, stream=self.stream)
        return y_recv

    def combine(self, y_perm, inv, tw):
        s = self.s
        out = torch.empty((int(s.T), int(s.d)), dtype=self.tdtype, device=self.device)
        B.combine(s, y_perm, inv, tw, out, stream=self.stream)
        return out

    def host_ints(self, t) -> np.ndarray:
        return t.cpu().numpy()

    def rows(self, n: int, like):
        return torch.empty((int(n),) + tuple(like.shape[1:]), dtype=like.dtype, device=like.device)

    def check(self):
        st = B.get_error(self.stream)
        if st != B.MOE_OK:
            raise B.MoEError(st, "expert-parallel forward")


def _bits(t: torch.Tensor) -> torch.Tensor:
    """The same rows as raw bytes [rows, row bytes] (transports need not know bf16)."""
    per_row = 1
    for n in t.shape[1:]:
        per_row *= int(n)
    if t.shape[0] == 0:                      # nothing to alias: a fresh empty block of the right width
        return torch.empty((0, per_row * t.element_size()), dtype=torch.uint8, device=t.device)
    return t.reshape(t.shape[0], per_row).view(torch.uint8)


def exchange_rows(t: torch.Tensor, send: np.ndarray, recv: np.ndarray, group, out: torch.Tensor) -> torch.Tensor:
    """All-to-all of row blocks: rank r's rows [sum(send[:g]), sum(send[:g+1]))
    go to rank g, and out receives rank g's block at [sum(recv[:g]), ...).
    Device tensors stay on the device for NCCL; with a host-only backend
    (gloo) they travel through host memory."""
    import torch.distributed as dist
    host = dist.get_backend(group) != "nccl" and t.is_cuda
    src = _bits(t.contiguous())
    dst = _bits(out)
    if host:
        src_h = src.cpu()
        dst_h = torch.empty(dst.shape, dtype=dst.dtype)
        dist.all_to_all_single(dst_h, src_h, [int(v) for v in recv], [int(v) for v in send], group=group)
        dst.copy_(dst_h)
    else:
        dist.all_to_all_single(dst, src, [int(v) for v in recv], [int(v) for v in send], group=group)
    return out


def exchange_counts(send_table: np.ndarray, group) -> np.ndarray:
    """All-to-all of the per-expert counts: rank r sends row g of its [G, E]
    table to rank g; returns the [G, E] table of what each source sends here."""
    import torch.distributed as dist
    G, E = send_table.shape
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    src = torch.from_numpy(np.ascontiguousarray(send_table, dtype=np.int64).reshape(-1)).to(dev)
    dst = torch.empty(G * E, dtype=torch.int64, device=dev)
    dist.all_to_all_single(dst, src, [E] * G, [E] * G, group=group)
    return dst.cpu().numpy().reshape(G, E)


def ep_forward(x, part: Partition, ops, group) -> dict:
    """The layer forward for this rank's tokens x with experts spread over the
    group's ranks. Returns dict(out, recv_counts, send_counts, routing...)."""
    import torch.distributed as dist
    G = dist.get_world_size(group)
    if G != part.G:
        raise ValueError(f"partition over {part.G} ranks, group has {G}")
    E = part.E
    r = ops.route_and_group(x)
    counts = ops.host_ints(r["counts"]).astype(np.int64)
    send = part.send_counts(counts)
    recv_counts = exchange_counts(counts.reshape(G, E), group)
    recv = recv_counts.sum(axis=1)
    recv_x = exchange_rows(r["x_perm"], send, recv, group, ops.rows(int(recv.sum()), r["x_perm"]))
    x_local, offsets_local, local_src = ops.regroup(G, E, recv_counts, recv_x)
    y_local = ops.ffn(x_local, offsets_local, E)
    y_recv = ops.ungroup(local_src, y_local)
    y_perm = exchange_rows(y_recv, recv, send, group, ops.rows(int(send.sum()), y_recv))
    out = ops.combine(y_perm, r["inv"], r["tw"])
    ops.check()
    return dict(out=out, counts=counts, send_counts=send, recv_counts=recv_counts,
                offsets_local=ops.host_ints(offsets_local), local_src=ops.host_ints(local_src),
                idx=r["idx"], tw=r["tw"])
