"""Expert capacity with token drop on the GPU against the oracle.

moe_permute_capacity must give the oracle's kept counts, offsets, perm,
inv_perm (with -2 for a dropped assignment) and drop count bit-exactly;
moe_forward_capacity must give the layer output of the oracle composed from
its own capacity grouping, FFN and combine (dropped assignments add nothing,
kept gate weights are not renormalised)."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import Inputs, dev, host_f64, new, oracle_outputs_for_tokens, rel_err, tol

pytestmark = pytest.mark.gpu


def gpu_permute_capacity(s, idx_h, x, cf, A, d, dtype):
    N = s.N
    counts, offsets = new((N,), "i32", fill=-1), new((N + 1,), "i32", fill=-1)
    perm, inv = new((max(A, 1),), "i32", fill=-7), new((max(A, 1),), "i32", fill=-7)
    xp = new((max(A, 1), d), dtype, fill=0)
    dropped = new((1,), "i32", fill=-1)
    ws = B.workspace(B.permute_workspace_size(s))
    B.permute_capacity(s, dev(idx_h) if A else None, x, cf, counts, offsets, perm, inv, xp, ws, dropped=dropped)
    assert B.get_error() == B.MOE_OK
    return counts, offsets, perm, inv, xp, dropped


@pytest.mark.parametrize("T,N,k,zipf", [(1, 4, 2, None), (300, 8, 2, None), (777, 32, 8, 1.2), (4096, 128, 8, 1.2),
                                        (5000, 64, 2, 1.5)])
@pytest.mark.parametrize("cf", [0.0, 0.25, 1.0, 1.25, 100.0])
def test_permute_capacity_bit_exact(T, N, k, zipf, cf):
    rng = np.random.default_rng(T * 7 + N)
    if zipf:
        p = 1.0 / np.arange(1, N + 1) ** zipf
        p /= p.sum()
    else:
        p = np.full(N, 1.0 / N)
    idx = np.stack([rng.choice(N, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    d = 128
    w = S.Workload("cap-x", T=T, d=d, N=1, k=1, F=64, act="swiglu", dtype="bf16", seed=T)
    x_h = S.x_all(w)
    s = B.shape(T, d, N, k, 64, "swiglu", "bf16")
    cap = oracle.capacity(T, N, k, cf)
    ref = oracle.permute_capacity(idx, N, cap)
    counts, offsets, perm, inv, xp, dropped = gpu_permute_capacity(s, idx, dev(x_h), cf, T * k, d, "bf16")
    np.testing.assert_array_equal(counts.cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(offsets.cpu().numpy(), ref["offsets"])
    kept = int(ref["offsets"][-1])
    np.testing.assert_array_equal(perm.cpu().numpy()[:kept], ref["perm"][:kept])
    np.testing.assert_array_equal(inv.cpu().numpy(), ref["inv_perm"])
    assert int(dropped.item()) == ref["dropped"]
    # kept rows carry their token's x
    if kept:
        assert torch.equal(xp[:kept], dev(x_h)[torch.from_numpy(ref["perm"][:kept]).long().cuda()])


def test_permute_capacity_empty_batch():
    s = B.shape(0, 128, 4, 2, 64, "swiglu", "bf16")
    counts, offsets, _, _, _, dropped = gpu_permute_capacity(s, np.zeros((0, 2), np.int32), None, 1.0, 0, 128,
                                                             "bf16")
    assert counts.cpu().tolist() == [0] * 4
    assert offsets.cpu().tolist() == [0] * 5
    assert int(dropped.item()) == 0


def test_permute_capacity_rejects_negative_factor():
    s = B.shape(4, 128, 4, 2, 64, "swiglu", "bf16")
    with pytest.raises(B.MoEError):
        gpu_permute_capacity(s, np.zeros((4, 2), np.int32), new((4, 128), "bf16", fill=0), -1.0, 8, 128, "bf16")


def oracle_forward_capacity(inp: Inputs, cf: float):
    """The oracle composed: route, capacity grouping, per-expert FFN of the
    kept rows, combine that skips dropped assignments."""
    w = inp.w
    r = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h)
    g = oracle.permute_capacity(r["topk_idx"], w.N, oracle.capacity(w.T, w.N, w.k, cf))
    y = np.zeros((w.A, w.d))
    xf = S.to_f64(inp.x_h, w.dtype)
    for e in range(w.N):
        a, b = g["offsets"][e], g["offsets"][e + 1]
        if b > a:
            rows = xf[g["perm"][a:b]]
            y[a:b] = oracle.expert_rows(rows, *inp.expert(e), w.act)
    out = oracle.combine(y, g["inv_perm"], r["topk_w"])
    return r, g, out


CAP_SMALL = [
    S.Workload("cap-swiglu", T=300, d=256, N=8, k=2, F=384, act="swiglu", dtype="bf16", seed=41),
    S.Workload("cap-skew-k8", T=256, d=256, N=32, k=8, F=192, act="swiglu", dtype="bf16", seed=42, zipf_s=1.2),
    S.Workload("cap-gelu-f32", T=100, d=64, N=6, k=3, F=96, act="gelu_tanh", dtype="f32", seed=43),
]


@pytest.mark.parametrize("cf", [0.5, 1.0, 1.25])
@pytest.mark.parametrize("w", CAP_SMALL, ids=[w.name for w in CAP_SMALL])
def test_forward_capacity_full_oracle(w, cf):
    inp = Inputs(w)
    s = inp.shape
    out = new((w.T, w.d), w.dtype, fill=0)
    idx = new((w.T, w.k), "i32")
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    cnt = new((w.N,), "i32")
    dropped = new((1,), "i32", fill=-1)
    ws = B.workspace(B.workspace_size(s))
    B.forward_capacity(s, cf, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws,
                       topk_idx=idx, topk_w=tw, counts=cnt, dropped=dropped)
    assert B.get_error() == B.MOE_OK
    r, g, ref = oracle_forward_capacity(inp, cf)
    np.testing.assert_array_equal(idx.cpu().numpy(), r["topk_idx"])
    np.testing.assert_array_equal(cnt.cpu().numpy(), g["counts"])
    assert int(dropped.item()) == g["dropped"]
    if cf < 1.0:
        assert g["dropped"] > 0                      # the case really drops
    assert rel_err(host_f64(out), ref) <= tol(w.dtype)


def test_forward_capacity_above_demand_equals_plain_forward():
    from tests.gpu_util import run_forward
    w = CAP_SMALL[1]
    inp = Inputs(w)
    plain = run_forward(inp)[0]
    s = inp.shape
    out = new((w.T, w.d), w.dtype)
    ws = B.workspace(B.workspace_size(s))
    B.forward_capacity(s, float(w.N), inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws)
    assert B.get_error() == B.MOE_OK
    assert torch.equal(out, plain)


def test_forward_capacity_full_size_zipf():
    """The skewed 16384-token, 128-expert, top-8 batch at capacity factor
    1.25: grouping bit-exact on every assignment, outputs of sampled tokens
    against the oracle (dropped assignments removed from their sum)."""
    w = S.WORKLOADS["zipf-skew-n128-k8"]
    cf = 1.25
    inp = Inputs(w, host_weights=False)
    s = inp.shape
    out = new((w.T, w.d), w.dtype)
    idx = new((w.T, w.k), "i32")
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    dropped = new((1,), "i32", fill=-1)
    ws = B.workspace(B.workspace_size(s))
    B.forward_capacity(s, cf, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws,
                       topk_idx=idx, topk_w=tw, dropped=dropped)
    assert B.get_error() == B.MOE_OK
    r = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h)
    np.testing.assert_array_equal(idx.cpu().numpy(), r["topk_idx"])
    g = oracle.permute_capacity(r["topk_idx"], w.N, oracle.capacity(w.T, w.N, w.k, cf))
    assert g["dropped"] > 0
    assert int(dropped.item()) == g["dropped"]
    tokens = np.sort(np.random.default_rng(2).choice(w.T, size=24, replace=False))
    kept = (g["inv_perm"].reshape(w.T, w.k) >= 0)
    tw_kept = np.where(kept, r["topk_w"], 0.0)       # a dropped assignment contributes nothing
    ref = oracle_outputs_for_tokens(inp, tokens, r["topk_idx"], tw_kept)
    got = host_f64(out[torch.from_numpy(tokens).cuda()])
    assert rel_err(got, ref) <= tol(w.dtype)
