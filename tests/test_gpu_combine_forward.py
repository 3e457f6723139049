"""moe_combine and the whole moe_forward against the oracle.

Small workloads run the full oracle layer; the full-size workloads (in the
launch configuration the benchmark times: route -> permute -> grouped FFN ->
combine on one stream) check routing, counts and the permutation bit-exactly
on every token and the outputs of sampled tokens against the oracle."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import (Inputs, check_route, dev, host_f64, new, oracle_outputs_for_tokens, rel_err,
                            run_forward, tol)

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- combine
@pytest.mark.parametrize("T,d,k,dtype", [(1, 128, 1, "bf16"), (300, 256, 2, "bf16"), (77, 512, 8, "bf16"),
                                         (64, 128, 2, "f32"), (9, 12, 3, "f32")])
def test_combine_matches_oracle(T, d, k, dtype):
    rng = np.random.default_rng(T + d)
    N = max(k, 8)
    idx = np.stack([rng.choice(N, k, replace=False) for _ in range(T)]).astype(np.int32)
    inv = oracle.permute(idx, N)["inv_perm"]
    w = rng.random((T, k)).astype(np.float32)
    w /= w.sum(1, keepdims=True)
    yw = S.Workload("comb", T=T * k, d=d, N=1, k=1, F=64, act="swiglu", dtype=dtype, seed=3)
    y_h = S.x_all(yw)
    s = B.shape(T, d, N, k, 64, "swiglu", dtype)
    out = new((T, d), dtype, fill=0)
    B.combine(s, dev(y_h), dev(inv), dev(w), out)
    assert B.get_error() == B.MOE_OK
    ref = oracle.combine(S.to_f64(y_h, dtype), inv, w.astype(np.float64))
    got = host_f64(out)
    assert rel_err(got, ref) <= tol(dtype)
    # one rounding to the output dtype on top of an fp32 sum: elementwise bound
    ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -23
    assert np.all(np.abs(got - ref) <= ulp * np.abs(ref) + 1e-5 * np.abs(ref).max() + 1e-30)


# ---------------------------------------------------------------- full layer, small
SMALL = [
    S.WORKLOADS["tiny-f32"],
    S.Workload("small-swiglu", T=300, d=256, N=8, k=2, F=384, act="swiglu", dtype="bf16", seed=21),
    S.Workload("small-gelu", T=257, d=384, N=16, k=2, F=256, act="gelu_tanh", dtype="bf16", seed=22),
    S.Workload("small-topk8-bias", T=200, d=256, N=32, k=8, F=192, act="swiglu", dtype="bf16", seed=23,
               zipf_s=1.2),
    S.Workload("one-token", T=1, d=128, N=4, k=2, F=128, act="swiglu", dtype="bf16", seed=24),
    S.Workload("k-equals-n", T=50, d=128, N=4, k=4, F=128, act="gelu_tanh", dtype="bf16", seed=25),
    S.Workload("f32-gelu", T=100, d=64, N=6, k=3, F=96, act="gelu_tanh", dtype="f32", seed=26),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_forward_small_full_oracle(w):
    inp = Inputs(w)
    out, idx, tw, cnt = run_forward(inp)
    WG = np.stack([inp.host[e][0] for e in range(w.N)])
    WU = np.stack([inp.host[e][1] for e in range(w.N)]) if w.act == "swiglu" else None
    WD = np.stack([inp.host[e][2] for e in range(w.N)])
    ref = oracle.forward(inp.x_h, inp.wg_h, inp.bias_h, WG, WU, WD, w.k, w.act)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_array_equal(cnt.cpu().numpy(), ref["counts"])
    np.testing.assert_allclose(tw.cpu().numpy(), ref["topk_w"], atol=1e-5)
    assert rel_err(host_f64(out), ref["out"]) <= tol(w.dtype)


def test_forward_repeatable_bitwise():
    inp = Inputs(SMALL[3])
    a = run_forward(inp)[0]
    b = run_forward(inp)[0]
    assert torch.equal(a, b)


def test_forward_empty_batch():
    w = S.Workload("empty", T=0, d=128, N=4, k=2, F=128, act="swiglu", dtype="bf16", seed=1)
    s = B.shape(0, 128, 4, 2, 128, "swiglu", "bf16")
    wg = torch.zeros(128, 4, device="cuda")
    W = torch.zeros(4, 128, 128, dtype=torch.bfloat16, device="cuda")
    cnt = new((4,), "i32", fill=-1)
    ws = B.workspace(B.workspace_size(s))
    B.forward(s, None, wg, None, W, W, W, None, ws, counts=cnt)
    assert B.get_error() == B.MOE_OK
    assert cnt.cpu().tolist() == [0, 0, 0, 0]


def test_forward_hostio_matches_device_forward():
    w = SMALL[1]
    inp = Inputs(w)
    out_dev = run_forward(inp)[0]
    s = inp.shape
    x_host = inp.x.cpu().pin_memory()
    out_host = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    ws = B.workspace(B.hostio_workspace_size(s))
    B.forward_hostio(s, x_host, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out_host, ws)
    torch.cuda.synchronize()
    assert B.get_error() == B.MOE_OK
    assert torch.equal(out_host, out_dev.cpu())


def test_forward_hostio_pipelined_matches_device_forward():
    """Consecutive batches through the three-stream pipelined call, slots
    alternating: every batch's host output equals the device forward's."""
    w = SMALL[1]
    inp = Inputs(w)
    s = inp.shape
    nb = 5
    xs = [(inp.x.float() * (1.0 + 0.25 * i)).to(torch.bfloat16) for i in range(nb)]
    refs = []
    for xb in xs:
        o = new((w.T, w.d), w.dtype)
        B.forward(s, xb, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, o, B.workspace(B.workspace_size(s)))
        refs.append(o)
    torch.cuda.synchronize()
    x_hosts = [xb.cpu().pin_memory() for xb in xs]
    outs = [torch.full((w.T, w.d), 7.0, dtype=torch.bfloat16).pin_memory() for _ in xs]
    ws = B.workspace(B.hostio_pipelined_workspace_size(s))
    comp, h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    for i in range(nb):
        B.forward_hostio_pipelined(s, x_hosts[i], inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, outs[i], ws,
                                   i % 2, comp, h2d, d2h)
    torch.cuda.synchronize()
    assert B.get_error() == B.MOE_OK
    for i in range(nb):
        assert torch.equal(outs[i], refs[i].cpu()), i


# ---------------------------------------------------------------- full size
def staged_forward(inp: Inputs):
    """The four C-ABI calls with every intermediate in caller buffers."""
    w, s = inp.w, inp.shape
    A = w.A
    idx, tw = new((w.T, w.k), "i32"), torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    counts, offsets = new((w.N,), "i32"), new((w.N + 1,), "i32")
    perm, inv = new((A,), "i32"), new((A,), "i32")
    xp, yp = new((A, w.d), w.dtype), new((A, w.d), w.dtype)
    out = new((w.T, w.d), w.dtype)
    ws = B.workspace(max(B.permute_workspace_size(s), B.grouped_ffn_workspace_size(s)))
    B.route(s, inp.x, inp.wg, inp.bias, idx, tw)
    B.permute(s, idx, inp.x, counts, offsets, perm, inv, xp, ws)
    B.grouped_ffn(s, xp, offsets, inp.w_gate, inp.w_up, inp.w_down, yp, ws)
    B.combine(s, yp, inv, tw, out)
    assert B.get_error() == B.MOE_OK
    return dict(idx=idx, tw=tw, counts=counts, offsets=offsets, perm=perm, inv=inv, xp=xp, yp=yp, out=out)


FULL = ["decode-t32-n64-k8", "prefill-n8-f14336", "zipf-skew-n128-k8", "worked-example-n64-f16384-gelu"]


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size(name):
    w = S.WORKLOADS[name]
    inp = Inputs(w, host_weights=False)
    r = staged_forward(inp)
    # routing: bit-exact on every token
    orc = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h)
    gi = r["idx"].cpu().numpy()
    check_route(gi, r["tw"].cpu().numpy().astype(np.float64), orc)
    # grouping: bit-exact
    pref = oracle.permute(gi, w.N)
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), pref["counts"])
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), pref["offsets"])
    np.testing.assert_array_equal(r["perm"].cpu().numpy(), pref["perm"])
    np.testing.assert_array_equal(r["inv"].cpu().numpy(), pref["inv_perm"])
    rows = np.random.default_rng(0).choice(w.A, size=min(w.A, 512), replace=False)
    assert torch.equal(r["xp"][torch.from_numpy(rows).cuda()],
                       inp.x[torch.from_numpy(pref["perm"][rows]).long().cuda()])
    # outputs of sampled tokens (every token for the decode batch)
    n_s = w.T if w.T <= 32 else 24
    tokens = np.sort(np.random.default_rng(1).choice(w.T, size=n_s, replace=False))
    ref = oracle_outputs_for_tokens(inp, tokens, orc["topk_idx"], orc["topk_w"])
    got = host_f64(r["out"][torch.from_numpy(tokens).cuda()])
    err = rel_err(got, ref)
    print(f"{name}: sampled-token max err / max|ref| = {err:.2e}")
    assert err <= tol(w.dtype)
    # the one-call forward gives the same bits as the staged calls
    out1 = run_forward(inp)[0]
    assert torch.equal(out1, r["out"])


def test_forward_captured_in_cuda_graph_replays_identically():
    """The forward only queues work on the caller's stream (no allocation, no
    host sync), so it can be captured once and replayed; the replay gives the
    same bits as a direct call, also after the inputs change in place."""
    w = SMALL[3]
    inp = Inputs(w)
    s = inp.shape
    out = new((w.T, w.d), w.dtype)
    ws = B.workspace(B.workspace_size(s))
    B.forward(s, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws)   # warm-up, outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            B.forward(s, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws)
    g.replay()
    torch.cuda.synchronize()
    direct = run_forward(inp)[0]
    assert torch.equal(out, direct)
    inp.x.mul_(-1.0)                                  # new inputs, same buffers
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, run_forward(inp)[0])
    assert B.get_error() == B.MOE_OK
