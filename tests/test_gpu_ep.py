"""Expert parallelism on the GPU: the regroup / ungroup kernels against the
oracle bit for bit, and the whole expert-parallel forward run by two
processes that share the one GPU, exchanging rows through a gloo group on the
host ("MoE混合专家模型计算原理与推理部署实战解析" section 3.3). Nothing here
waits on another process's kernels: each exchange is a host collective
between complete kernel launches."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from mixture_experts_layer_97_b300 import ep

pytestmark = pytest.mark.gpu


def _table(seed, G, E, empty_frac=0.3, hi=40):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, hi, size=(G, E)) * (rng.random((G, E)) >= empty_frac)).astype(np.int32)


@pytest.mark.parametrize("G,E,d,dtype", [(2, 4, 256, "bf16"), (4, 16, 128, "bf16"), (8, 32, 64, "f32"),
                                         (1, 1, 8, "bf16"), (16, 16, 384, "bf16")])
def test_regroup_and_ungroup_match_the_oracle(G, E, d, dtype):
    rc = _table(G * 100 + E, G, E)
    rows = int(rc.sum())
    ref = oracle.ep_regroup(rc)
    td = B.TORCH_DTYPE[dtype]
    recv_x = torch.randn(rows, d, device="cuda").to(td)
    x_local = torch.zeros_like(recv_x)
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    src = torch.full((rows,), -1, dtype=torch.int32, device="cuda")
    B.ep_regroup(G, E, torch.from_numpy(rc).cuda(), recv_x, x_local, off, src, dtype)
    assert B.get_error() == B.MOE_OK
    np.testing.assert_array_equal(off.cpu().numpy(), ref["offsets_local"])
    np.testing.assert_array_equal(src.cpu().numpy(), ref["local_src"])
    assert torch.equal(x_local, recv_x[src.long()])
    y_recv = torch.zeros_like(x_local)
    B.ep_ungroup(src, x_local, y_recv, dtype)
    assert B.get_error() == B.MOE_OK
    assert torch.equal(y_recv, recv_x)                   # ungroup inverts regroup


def test_regroup_records_a_table_that_does_not_add_up():
    rc = np.array([[3, 2], [1, 0]], dtype=np.int32)
    recv_x = torch.zeros(5, 128, dtype=torch.bfloat16, device="cuda")     # the table says 6 rows
    out = torch.zeros_like(recv_x)
    off = torch.full((3,), -1, dtype=torch.int32, device="cuda")
    src = torch.full((5,), -1, dtype=torch.int32, device="cuda")
    B.ep_regroup(2, 2, torch.from_numpy(rc).cuda(), recv_x, out, off, src, "bf16")
    assert B.get_error() == B.MOE_ERR_CORRUPT
    assert int(off[0].item()) == -1                      # nothing written


def test_regroup_rejects_bad_arguments():
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoEError):
        B.ep_regroup(16, 17, i, x, x, i, i, "bf16")        # G * E > 256
    y = torch.zeros(4, 4, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MoEError):
        B.ep_regroup(1, 1, i, y, y, i, i, "bf16")          # 8-byte rows: not a multiple of 16


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


W_EP = S.Workload("ep-gpu", T=300, d=256, N=8, k=2, F=384, act="swiglu", dtype="bf16", seed=81, zipf_s=1.2)


def _rank_tokens(rank):
    T = W_EP.T + 37 * rank
    lo = sum(W_EP.T + 37 * r for r in range(rank))
    return S.x_rows(W_EP.scaled(T=4096), lo, lo + T)


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        w = W_EP
        x_h = _rank_tokens(rank)
        T = x_h.shape[0]
        part = ep.Partition(w.N, world)
        dev = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
                         else torch.from_numpy(a)).cuda()
        mine = list(part.experts(rank))
        ex = {e: S.expert_weights(w, e) for e in range(w.N)}
        WG = dev(np.stack([ex[e][0] for e in mine]))
        WU = dev(np.stack([ex[e][1] for e in mine]))
        WD = dev(np.stack([ex[e][2] for e in mine]))
        wg_h, b_h = S.gate_weight(w), S.gate_bias(w)
        s = B.shape(T, w.d, w.N, w.k, w.F, w.act, w.dtype)
        ops = ep.CudaOps(s, w.dtype, dev(wg_h), dev(b_h), WG, WU, WD)
        res = ep.ep_forward(dev(x_h), part, ops, group=dist.group.WORLD)
        torch.cuda.synchronize()
        got = res["out"].float().cpu().numpy().astype(np.float64)
        # the single-process oracle layer with all experts on this rank's tokens
        A = lambda i: np.stack([ex[e][i] for e in range(w.N)])
        ref = oracle.forward(x_h, wg_h, b_h, A(0), A(1), A(2), w.k, w.act)
        err = float(np.abs(got - ref["out"]).max() / np.abs(ref["out"]).max())
        # the same tokens through the one-GPU forward of the library (all experts)
        s_all = B.shape(T, w.d, w.N, w.k, w.F, w.act, w.dtype)
        one = torch.empty(T, w.d, dtype=torch.bfloat16, device="cuda")
        B.forward(s_all, dev(x_h), dev(wg_h), dev(b_h), dev(A(0)), dev(A(1)), dev(A(2)), one,
                  B.workspace(B.workspace_size(s_all)))
        torch.cuda.synchronize()
        err_one = float((res["out"].float() - one.float()).abs().max().item() / one.float().abs().max().item())
        out[rank] = dict(err=err, err_one=err_one, idx_ok=bool(np.array_equal(res["idx"].cpu().numpy(),
                                                                              ref["topk_idx"])),
                         counts=res["counts"].tolist(), ref_counts=ref["counts"].tolist(),
                         recv_counts=res["recv_counts"].tolist(), offsets_local=res["offsets_local"].tolist(),
                         status=B.get_error())
    finally:
        dist.destroy_process_group()


def test_expert_parallel_forward_two_processes_on_one_gpu():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    E = W_EP.N // world
    for r in range(world):
        print(f"rank {r}: EP forward vs oracle {res[r]['err']:.2e}, vs one-GPU forward {res[r]['err_one']:.2e}")
        assert res[r]["status"] == B.MOE_OK
        assert res[r]["idx_ok"]
        assert res[r]["counts"] == res[r]["ref_counts"]
        assert res[r]["err"] <= 2e-2
        assert res[r]["err_one"] <= 2e-2
    for g in range(world):
        ref_rc = np.array([res[r]["counts"][g * E:(g + 1) * E] for r in range(world)], dtype=np.int32)
        assert res[g]["recv_counts"] == ref_rc.tolist()
        assert res[g]["offsets_local"] == oracle.ep_regroup(ref_rc)["offsets_local"].tolist()
