"""Selection-only expert bias and routing statistics on the GPU against the oracle.

moe_route_ex with MOE_BIAS_SELECT must choose the oracle's experts bit-exactly
(the choosing score is the fp32 sum logit + bias on both sides) and give its
weights within 1e-5; the load statistics must match the oracle's
load_stats computed on the same routing:
  f: exact up to the float rounding of count / (T k)   (rel 1e-6)
  P, N sum f P, mean top-1: fp32 softmax summed per CTA, then fp64   (rel 1e-5)
  entropy (bits): from f                                              (abs 1e-5)
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import Inputs, check_route, dev, host_f64, new, rel_err, run_forward, tol

pytestmark = pytest.mark.gpu

TOL_STATS = 1e-5


def gpu_route_ex(inp, bias_mode, stats=True):
    w = inp.w
    s = inp.shape
    idx = new((w.T, w.k), "i32", fill=-1)
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    st = torch.full((B.load_stats_len(w.N),), -1.0, dtype=torch.float32, device="cuda") if stats else None
    ws = B.workspace(B.route_ex_workspace_size(s)) if stats else None
    B.route_ex(s, inp.x, inp.wg, inp.bias, idx, tw, bias_mode=bias_mode, load_stats=st, ws=ws)
    assert B.get_error() == B.MOE_OK
    return idx, tw, st


def check_stats(st_gpu, N, probs, idx):
    ref = oracle.load_stats(probs, idx)
    got = B.unpack_load_stats(st_gpu, N)
    np.testing.assert_allclose(got["f"], ref["f"], rtol=1e-6, atol=0)
    np.testing.assert_allclose(got["P"], ref["P"], rtol=TOL_STATS, atol=1e-7)
    assert got["balance"] == pytest.approx(ref["balance"], rel=TOL_STATS)
    assert got["entropy_bits"] == pytest.approx(ref["entropy_bits"], abs=1e-5)
    assert got["top1"] == pytest.approx(ref["top1"], rel=TOL_STATS)
    return got


BIASED = [
    S.Workload("sel-small", T=300, d=256, N=16, k=2, F=128, act="swiglu", dtype="bf16", seed=51, zipf_s=1.2),
    S.Workload("sel-k8", T=777, d=384, N=64, k=8, F=128, act="swiglu", dtype="bf16", seed=52, zipf_s=1.2),
    S.Workload("sel-few-experts", T=1000, d=128, N=8, k=2, F=128, act="swiglu", dtype="bf16", seed=53, zipf_s=1.5),
    S.Workload("sel-f32", T=99, d=64, N=6, k=3, F=96, act="gelu_tanh", dtype="f32", seed=54, zipf_s=1.2),
    S.Workload("sel-n256", T=64, d=128, N=256, k=4, F=128, act="swiglu", dtype="bf16", seed=55, zipf_s=1.2),
]


@pytest.mark.parametrize("mode", ["select", "logits"])
@pytest.mark.parametrize("w", BIASED, ids=[w.name for w in BIASED])
def test_route_ex_matches_oracle(w, mode):
    inp = Inputs(w, host_weights=False)
    idx, tw, st = gpu_route_ex(inp, mode)
    orc = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h, bias_mode=mode, want_probs=True)
    check_route(idx.cpu().numpy(), tw.cpu().numpy().astype(np.float64), orc)
    check_stats(st, w.N, orc["probs"], orc["topk_idx"])


def test_select_mode_changes_weights_not_only_choice():
    """On the skewed bias the two modes choose the same experts per token
    (same score) but weight them differently."""
    w = BIASED[0]
    inp = Inputs(w, host_weights=False)
    i_sel, w_sel, _ = gpu_route_ex(inp, "select", stats=False)
    i_log, w_log, _ = gpu_route_ex(inp, "logits", stats=False)
    assert torch.equal(i_sel, i_log)
    assert not torch.allclose(w_sel, w_log)


def test_statistics_do_not_change_the_routing():
    w = BIASED[1]
    inp = Inputs(w, host_weights=False)
    a = gpu_route_ex(inp, "logits", stats=True)
    b = gpu_route_ex(inp, "logits", stats=False)
    idx = new((w.T, w.k), "i32")
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    B.route(inp.shape, inp.x, inp.wg, inp.bias, idx, tw)
    for got in (a, b):
        assert torch.equal(got[0], idx) and torch.equal(got[1], tw)


def test_statistics_repeatable_bitwise():
    inp = Inputs(BIASED[1], host_weights=False)
    assert torch.equal(gpu_route_ex(inp, "select")[2], gpu_route_ex(inp, "select")[2])


def test_statistics_uniform_gate():
    """W_g = 0: every probability is 1/N (top-1 1/N) and, with k = N, every
    expert takes every token: f = 1/N, N sum f P = 1, entropy log2 N."""
    N = 16
    s = B.shape(200, 128, N, N, 64, "swiglu", "bf16")
    x = new((200, 128), "bf16", fill=1.0)
    wg = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    idx = new((200, N), "i32")
    tw = torch.empty((200, N), dtype=torch.float32, device="cuda")
    st = torch.empty(B.load_stats_len(N), dtype=torch.float32, device="cuda")
    B.route_ex(s, x, wg, None, idx, tw, load_stats=st, ws=B.workspace(B.route_ex_workspace_size(s)))
    assert B.get_error() == B.MOE_OK
    g = B.unpack_load_stats(st, N)
    np.testing.assert_allclose(g["f"], 1.0 / N, rtol=1e-6)
    np.testing.assert_allclose(g["P"], 1.0 / N, rtol=1e-6)
    assert g["balance"] == pytest.approx(1.0, rel=1e-6)
    assert g["entropy_bits"] == pytest.approx(4.0, abs=1e-6)
    assert g["top1"] == pytest.approx(1.0 / N, rel=1e-6)


def test_statistics_empty_batch():
    s = B.shape(0, 128, 8, 2, 64, "swiglu", "bf16")
    st = torch.full((B.load_stats_len(8),), 5.0, dtype=torch.float32, device="cuda")
    wg = torch.zeros((128, 8), dtype=torch.float32, device="cuda")
    B.route_ex(s, None, wg, None, None, None, load_stats=st, ws=None)
    assert B.get_error() == B.MOE_OK
    assert float(st.abs().max()) == 0.0


def test_route_ex_rejects_bad_mode():
    s = B.shape(4, 128, 8, 2, 64, "swiglu", "bf16")
    L = B.lib()
    st = L.moe_route_ex(B.ctypes.byref(s), None, None, None, 7, None, None, None, None, 0, None)
    assert st == B.MOE_ERR_INVALID_ARG


def test_route_ex_full_size_zipf_select():
    """The skewed 16384-token, 128-expert, top-8 batch with the bias used for
    selection only: bit-exact choice on every token, statistics as the oracle."""
    w = S.WORKLOADS["zipf-skew-n128-k8"]
    inp = Inputs(w, host_weights=False)
    idx, tw, st = gpu_route_ex(inp, "select")
    orc = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h, bias_mode="select", want_probs=True)
    check_route(idx.cpu().numpy(), tw.cpu().numpy().astype(np.float64), orc)
    g = check_stats(st, w.N, orc["probs"], orc["topk_idx"])
    print(f"zipf select: balance {g['balance']:.3f}, entropy {g['entropy_bits']:.3f} bits, top1 {g['top1']:.3f}")


# ---------------------------------------------------------------- forward with options
OPT = [
    S.Workload("opt-swiglu", T=300, d=256, N=8, k=2, F=384, act="swiglu", dtype="bf16", seed=61, zipf_s=1.2),
    S.Workload("opt-k8", T=256, d=256, N=32, k=8, F=192, act="swiglu", dtype="bf16", seed=62, zipf_s=1.2),
]


@pytest.mark.parametrize("cf", [None, 0.75])
@pytest.mark.parametrize("w", OPT, ids=[w.name for w in OPT])
def test_forward_ex_select_bias_capacity_stats(w, cf):
    inp = Inputs(w)
    s = inp.shape
    out = new((w.T, w.d), w.dtype, fill=0)
    idx = new((w.T, w.k), "i32")
    st = torch.empty(B.load_stats_len(w.N), dtype=torch.float32, device="cuda")
    dropped = new((1,), "i32", fill=-1)
    ws = B.workspace(B.workspace_size(s))
    B.forward_ex(s, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws, bias_mode="select",
                 capacity_factor=cf, load_stats=st, dropped=dropped, topk_idx=idx)
    assert B.get_error() == B.MOE_OK
    r = oracle.route(inp.x_h, inp.wg_h, w.k, bias=inp.bias_h, bias_mode="select", want_probs=True)
    np.testing.assert_array_equal(idx.cpu().numpy(), r["topk_idx"])
    check_stats(st, w.N, r["probs"], r["topk_idx"])
    cap = oracle.capacity(w.T, w.N, w.k, cf) if cf is not None else w.A
    g = oracle.permute_capacity(r["topk_idx"], w.N, cap)
    assert int(dropped.item()) == g["dropped"]
    xf = S.to_f64(inp.x_h, w.dtype)
    y = np.zeros((w.A, w.d))
    for e in range(w.N):
        a, b = g["offsets"][e], g["offsets"][e + 1]
        if b > a:
            y[a:b] = oracle.expert_rows(xf[g["perm"][a:b]], *inp.expert(e), w.act)
    ref = oracle.combine(y, g["inv_perm"], r["topk_w"])
    assert rel_err(host_f64(out), ref) <= tol(w.dtype)


def test_forward_ex_without_options_is_the_plain_forward():
    w = OPT[0]
    inp = Inputs(w)
    plain = run_forward(inp)[0]
    out = new((w.T, w.d), w.dtype)
    B.forward_ex(inp.shape, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out,
                 B.workspace(B.workspace_size(inp.shape)))
    assert B.get_error() == B.MOE_OK
    assert torch.equal(out, plain)


def test_forward_ex_per_call_tiling_leaves_the_process_setting_alone():
    """A per-call tiling gives, bit for bit, what the same tiling set process
    wide gives, and does not change the process-wide setting."""
    w = S.Workload("tiling-call", T=600, d=512, N=4, k=2, F=384, act="swiglu", dtype="bf16", seed=63)
    inp = Inputs(w)
    s = inp.shape
    ws = B.workspace(B.workspace_size(s))
    outs = {}
    for mode in ("rows", "tokens", "pairs"):
        B.set_ffn_tiling(mode)
        outs[mode] = run_forward(inp)[0]
    B.set_ffn_tiling("auto")
    for mode in ("rows", "tokens", "pairs"):
        out = new((w.T, w.d), w.dtype)
        B.forward_ex(s, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws, ffn_tiling=mode)
        assert B.get_error() == B.MOE_OK
        assert torch.equal(out, outs[mode]), mode
        assert B.get_ffn_tiling() == "auto"
