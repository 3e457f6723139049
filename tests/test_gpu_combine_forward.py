"""moe_combine and the whole moe_forward against the oracle.

Small workloads run the full oracle layer; the full-size workloads (in the
launch configuration the benchmark times: route -> permute -> grouped FFN ->
combine on one stream) check routing, counts and the permutation bit-exactly
on every token, h and y_perm on a row set that holds every tile block of the
grouped GEMMs, and the outputs of every token (decode, skewed batch) or of
at least one token per expert (prefill, worked example)."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests import tiles
from tests.gpu_util import Inputs, check_route, dev, host_f64, new, rel_err, run_forward, tol

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
    return dict(idx=idx, tw=tw, counts=counts, offsets=offsets, perm=perm, inv=inv, xp=xp, yp=yp, out=out, ws=ws)


FULL = ["decode-t32-n64-k8", "prefill-n8-f14336", "zipf-skew-n128-k8", "worked-example-n64-f16384-gelu"]
# every output row compared where the oracle finishes the whole batch in about a minute
WHOLE_BATCH = {"decode-t32-n64-k8", "zipf-skew-n128-k8"}


def _h_rows(ws: torch.Tensor, rows: np.ndarray, A: int, F: int) -> torch.Tensor:
    """Rows of the hidden activations h [A, F] (bf16) that moe_grouped_ffn
    leaves at the start of its workspace."""
    h = ws[:A * F * 2].view(torch.bfloat16).view(A, F)
    return h[torch.from_numpy(rows).cuda()]


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size(name):
    """Full-size parity in the launch configuration the benchmark times.

    - top-k indices, counts, offsets, perm and inv_perm: bit-exact on every token;
    - x_perm: every row equals x[perm[row]];
    - h and y_perm: element by element against the oracle's expert FFN on a
      stratified row set that holds at least one row of every block of both
      grouped-GEMM tilings (asserted from offsets), over all columns;
    - out: every token on the decode and skewed batches (the whole y_perm
      too), else at least one token per active expert.
    """
    w = S.WORKLOADS[name]
    x_h, wg_h, bias_h = S.x_all(w), S.gate_weight(w), S.gate_bias(w)
    orc = oracle.route(x_h, wg_h, w.k, bias=bias_h)
    pref = oracle.permute(orc["topk_idx"], w.N)
    counts, offsets, perm = pref["counts"], pref["offsets"], pref["perm"]
    strat = tiles.stratified_rows(offsets)
    assert tiles.uncovered(counts, offsets, strat) == []
    whole = name in WHOLE_BATCH
    if whole:
        out_tokens = np.arange(w.T)
    else:   # the token of every active expert's first row, and of its last
        firsts = [int(perm[offsets[e]]) for e in range(w.N) if counts[e] > 0]
        lasts = [int(perm[offsets[e + 1] - 1]) for e in range(w.N) if counts[e] > 0]
        out_tokens = np.unique(firsts + lasts)
    out_rows = pref["inv_perm"].reshape(w.T, w.k)[out_tokens].reshape(-1)
    y_rows = np.arange(w.A) if whole else np.union1d(strat, out_rows)

    # oracle expert FFN on the needed rows, computed while the weights are uploaded
    y_ref = np.zeros((w.A, w.d)) if whole else {}
    h_ref = {}
    strat_set = set(strat.tolist())

    def on_expert(e, ws3):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows = y_rows[(y_rows >= lo) & (y_rows < hi)]
        if rows.size == 0:
            return
        y, h = oracle.expert_rows(x_h[perm[rows]], ws3[0], ws3[1], ws3[2], w.act, want_h=True)
        for i, r in enumerate(rows.tolist()):
            y_ref[r] = y[i]
            if r in strat_set:
                h_ref[r] = h[i]

    inp = Inputs(w, host_weights=False, on_expert=on_expert)
    r = staged_forward(inp)

    # routing and grouping: bit-exact
    check_route(r["idx"].cpu().numpy(), r["tw"].cpu().numpy().astype(np.float64), orc)
    np.testing.assert_array_equal(r["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(r["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(r["perm"].cpu().numpy(), perm)
    np.testing.assert_array_equal(r["inv"].cpu().numpy(), pref["inv_perm"])
    assert torch.equal(r["xp"], inp.x[r["perm"].long()])

    # h and y_perm on the stratified rows (every block of both tilings)
    hs = host_f64(_h_rows(r["ws"], strat, w.A, w.F))
    h_err = rel_err(hs, np.stack([h_ref[q] for q in strat.tolist()]))
    ys = host_f64(r["yp"][torch.from_numpy(strat).cuda()])
    y_err = rel_err(ys, np.stack([y_ref[q] for q in strat.tolist()]))
    # out on the chosen tokens
    if whole:
        y_full = y_ref
    else:
        y_full = np.zeros((w.A, w.d))
        for q in out_rows.tolist():
            y_full[q] = y_ref[q]
    out_ref = oracle.combine(y_full, pref["inv_perm"], orc["topk_w"], tokens=out_tokens)
    out_err = rel_err(host_f64(r["out"][torch.from_numpy(out_tokens).cuda()]), out_ref)
    n_units = len(tiles.units(counts))
    msg = (f"{name}: {len(strat)} stratified rows over {n_units} tile blocks of {int((counts > 0).sum())} experts, "
           f"{len(out_tokens)} output tokens; max err / max|ref|: h {h_err:.2e}, y_perm {y_err:.2e}, out {out_err:.2e}")
    if whole:
        yall_err = rel_err(host_f64(r["yp"]), y_ref)
        msg += f", whole y_perm {yall_err:.2e}"
        assert yall_err <= tol(w.dtype)
    print(msg)
    assert h_err <= tol(w.dtype)
    assert y_err <= tol(w.dtype)
    assert out_err <= tol(w.dtype)
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
