"""Expert parallelism on the host: the orchestration of
mixture_experts_layer_97_b300.ep (count exchange, row all-to-all, regroup,
local experts, ungroup, reverse all-to-all, combine) run by 1, 2, 4 and 8
gloo ranks, each step computed by the CPU oracle. Every rank's output must equal,
bit for bit in fp64, the single-process oracle forward of that rank's tokens
with all N experts ("MoE混合专家模型计算原理与推理部署实战解析" section 3.3:
splitting the experts over cards changes where a row is computed, not what)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import ep


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_workload(rank: int) -> S.Workload:
    # same layer (gate, experts: one seed) on every rank; each rank its own tokens
    return S.Workload("ep-host", T=40 + 13 * rank, d=64, N=8, k=2, F=48, act="swiglu", dtype="bf16", seed=71,
                      zipf_s=1.2)


def _rank_main(rank, world, port, out):
    from tests.ep_oracle_ops import OracleOps, _t
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = rank_workload(rank)
        # tokens of this rank: rows of a larger seeded batch, disjoint per rank
        big = w.scaled(T=1000)
        lo = sum(rank_workload(r).T for r in range(rank))
        x = S.x_rows(big, lo, lo + w.T)
        part = ep.Partition(w.N, world)
        res = ep.ep_forward(_t(x), part, OracleOps(w, rank, part), group=dist.group.WORLD)
        WG, WU, WD = (np.stack([S.expert_weights(w, e)[i] for e in range(w.N)]) for i in range(3))
        ref = oracle.forward(x, S.gate_weight(w), S.gate_bias(w), WG, WU, WD, w.k, w.act)
        out[rank] = dict(equal=bool(np.array_equal(res["out"].numpy(), ref["out"])),
                         counts=ref["counts"].tolist(), got_counts=res["counts"].tolist(),
                         recv_counts=res["recv_counts"].tolist(), send=res["send_counts"].tolist(),
                         offsets_local=res["offsets_local"].tolist())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [1, 2, 4, 8])
def test_expert_parallel_forward_equals_single_process_oracle(world):
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    E = 8 // world
    for r in range(world):
        assert res[r]["equal"], f"rank {r}"
        assert res[r]["got_counts"] == res[r]["counts"]
        assert res[r]["send"] == [sum(res[r]["counts"][g * E:(g + 1) * E]) for g in range(world)]
    # what rank g received from rank r is exactly what r counted for g's experts
    for g in range(world):
        for r in range(world):
            assert res[g]["recv_counts"][r] == res[r]["counts"][g * E:(g + 1) * E]
        assert res[g]["offsets_local"][-1] == sum(sum(res[r]["counts"][g * E:(g + 1) * E]) for r in range(world))


def test_partition_rejects_uneven_split():
    with pytest.raises(ValueError):
        ep.Partition(10, 4)
    p = ep.Partition(8, 4)
    assert list(p.experts(3)) == [6, 7]
    assert p.send_counts(np.arange(8)).tolist() == [1, 5, 9, 13]
