"""Expert-choice routing and the expert-choice layer on the GPU.

The choice is an integer decision taken on fp32 probabilities, so it is
checked two ways:
  - bit-exactly against its definition applied to the kernel's own fp32
    probabilities (top-C per expert by (p descending, token ascending), rows
    in ascending token order, inv / w the inverse tables);
  - against the oracle (fp64 softmax of the same fp32 logits): the chosen
    sets agree except for tokens whose oracle probability lies within the
    fp32 error bound of the expert's threshold (several choices are then
    correct; the kernel's must be one of them).
The probabilities themselves match the oracle within that bound, and the
layer output matches the oracle composed on the kernel's (validated) choice:
out[t] = sum over the experts e that picked t of p[t,e] * FFN_e(x_t).
"""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import Inputs, host_f64, new, rel_err, tol

pytestmark = pytest.mark.gpu


def p_bound(N):
    """Relative error bound of an fp32 softmax value (exp, an N-term sum, one
    division, one product), doubled for safety."""
    return (N + 8) * 2.0 ** -23


def gpu_route_ec(inp, C):
    w = inp.w
    s = inp.shape
    T, N = w.T, w.N
    probs = torch.full((max(T, 1), N), -1.0, dtype=torch.float32, device="cuda")
    perm = new((max(N * C, 1),), "i32", fill=-7)
    counts, offsets = new((N,), "i32", fill=-1), new((N + 1,), "i32", fill=-1)
    inv = new((max(T, 1), N), "i32", fill=-7)
    wt = torch.full((max(T, 1), N), -1.0, dtype=torch.float32, device="cuda")
    B.route_expert_choice(s, C, inp.x if T else None, inp.wg, inp.bias, probs, perm, counts, offsets, inv, wt)
    assert B.get_error() == B.MOE_OK
    return dict(probs=probs[:T].cpu().numpy(), perm=perm[:N * C].cpu().numpy(), counts=counts.cpu().numpy(),
                offsets=offsets.cpu().numpy(), inv=inv[:T].cpu().numpy(), w=wt[:T].cpu().numpy())


def check_definition(g, T, N, C):
    """The kernel's choice is the definition applied to its own fp32 probs."""
    p = g["probs"]
    assert g["counts"].tolist() == [C] * N
    assert g["offsets"].tolist() == [e * C for e in range(N + 1)]
    for e in range(N):
        want = np.sort(np.lexsort((np.arange(T), -p[:, e].astype(np.float64)))[:C])
        np.testing.assert_array_equal(g["perm"][e * C:(e + 1) * C], want)
        col = g["inv"][:, e]
        rows = np.full(T, -2, np.int32)
        rows[want] = e * C + np.arange(C)
        np.testing.assert_array_equal(col, rows)
        wcol = np.zeros(T, np.float32)
        wcol[want] = p[want, e]
        np.testing.assert_array_equal(g["w"][:, e], wcol)


def check_against_oracle(g, orc_probs, C):
    T, N = orc_probs.shape
    np.testing.assert_allclose(g["probs"], orc_probs, rtol=p_bound(N), atol=1e-30)
    ref = oracle.expert_choice(orc_probs, C)
    fragile = 0
    for e in range(N):
        a = set(g["perm"][e * C:(e + 1) * C].tolist())
        b = set(ref["perm"][e * C:(e + 1) * C].tolist())
        thr = ref["thr"][e]
        for t in a ^ b:
            assert abs(orc_probs[t, e] - thr) <= 2 * p_bound(N) * thr, (e, t)
            fragile += 1
    return fragile


ROUTE_CASES = [
    (S.Workload("ec-small", T=300, d=256, N=8, k=2, F=64, act="swiglu", dtype="bf16", seed=71), 75),
    (S.Workload("ec-ragged", T=1000, d=384, N=64, k=2, F=64, act="swiglu", dtype="bf16", seed=72), 31),
    (S.Workload("ec-bias", T=777, d=128, N=16, k=2, F=64, act="swiglu", dtype="bf16", seed=73, zipf_s=1.2), 100),
    (S.Workload("ec-all", T=50, d=128, N=4, k=2, F=64, act="swiglu", dtype="bf16", seed=74), 50),
    (S.Workload("ec-one", T=3000, d=128, N=32, k=2, F=64, act="swiglu", dtype="bf16", seed=75), 1),
    (S.Workload("ec-f32", T=99, d=64, N=6, k=3, F=96, act="gelu_tanh", dtype="f32", seed=76), 40),
    (S.Workload("ec-n256", T=2100, d=128, N=256, k=2, F=64, act="swiglu", dtype="bf16", seed=77), 2048),
]


@pytest.mark.parametrize("w,C", ROUTE_CASES, ids=[c[0].name for c in ROUTE_CASES])
def test_route_expert_choice(w, C):
    inp = Inputs(w, host_weights=False)
    g = gpu_route_ec(inp, C)
    check_definition(g, w.T, w.N, C)
    orc = oracle.route(inp.x_h, inp.wg_h, 1, bias=inp.bias_h, want_probs=True)
    n = check_against_oracle(g, orc["probs"], C)
    print(f"{w.name}: {n} near-threshold choices differ from the oracle's")


def test_route_expert_choice_exact_ties_take_lower_tokens():
    """W_g = 0: every probability is exactly 1/N, all tokens tie; each expert
    must take tokens 0 .. C-1."""
    T, N, C = 2500, 8, 1100
    s = B.shape(T, 128, N, 2, 64, "swiglu", "bf16")
    x = torch.ones((T, 128), dtype=torch.bfloat16, device="cuda")
    wg = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    probs = torch.empty((T, N), dtype=torch.float32, device="cuda")
    perm, counts, offsets = new((N * C,), "i32"), new((N,), "i32"), new((N + 1,), "i32")
    inv, wt = new((T, N), "i32"), torch.empty((T, N), dtype=torch.float32, device="cuda")
    B.route_expert_choice(s, C, x, wg, None, probs, perm, counts, offsets, inv, wt)
    assert B.get_error() == B.MOE_OK
    assert torch.all(probs == 1.0 / N)
    np.testing.assert_array_equal(perm.cpu().numpy(), np.tile(np.arange(C), N))


def test_route_expert_choice_rejects_capacity_above_tokens():
    s = B.shape(10, 128, 4, 2, 64, "swiglu", "bf16")
    assert B.lib().moe_route_expert_choice(B.ctypes.byref(s), 11, None, None, None, None, None, None, None, None,
                                           None, None) == B.MOE_ERR_INVALID_ARG
    assert B.expert_choice_workspace_size(s, 11) == 0


def ec_reference(inp, g, tokens=None):
    """Oracle layer output on the kernel's validated choice, with the
    oracle's probabilities as the weights."""
    w = inp.w
    orc = oracle.route(inp.x_h, inp.wg_h, 1, bias=inp.bias_h, want_probs=True)
    p = orc["probs"]
    tokens = np.arange(w.T) if tokens is None else np.asarray(tokens)
    xf = S.to_f64(inp.x_h, w.dtype)
    out = np.zeros((len(tokens), w.d))
    for e in range(w.N):
        q = np.nonzero(g["inv"][tokens, e] >= 0)[0]
        if len(q):
            out[q] += p[tokens[q], e][:, None] * oracle.expert_rows(xf[tokens[q]], *inp.expert(e), w.act)
    return out


FWD_CASES = [
    (S.Workload("ecf-swiglu", T=300, d=256, N=8, k=2, F=384, act="swiglu", dtype="bf16", seed=81), 75),
    (S.Workload("ecf-gelu-ragged", T=257, d=384, N=16, k=2, F=256, act="gelu_tanh", dtype="bf16", seed=82), 33),
    (S.Workload("ecf-f32", T=100, d=64, N=6, k=3, F=96, act="gelu_tanh", dtype="f32", seed=83), 50),
    (S.Workload("ecf-none", T=64, d=128, N=4, k=2, F=128, act="swiglu", dtype="bf16", seed=84), 0),
]


@pytest.mark.parametrize("w,C", FWD_CASES, ids=[c[0].name for c in FWD_CASES])
def test_forward_expert_choice(w, C):
    inp = Inputs(w)
    s = inp.shape
    g = gpu_route_ec(inp, C)
    out = new((w.T, w.d), w.dtype, fill=7)
    counts = new((w.N,), "i32", fill=-1)
    ws = B.workspace(B.expert_choice_workspace_size(s, C))
    B.forward_expert_choice(s, C, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws, counts=counts)
    assert B.get_error() == B.MOE_OK
    assert counts.cpu().tolist() == [C] * w.N
    got = host_f64(out)
    if C == 0:
        assert np.all(got == 0.0)                    # picked by no expert: the layer adds nothing
        return
    ref = ec_reference(inp, g)
    assert rel_err(got, ref) <= tol(w.dtype)
    unpicked = np.all(g["inv"] < 0, axis=1)
    assert np.all(got[unpicked] == 0.0)


def test_forward_expert_choice_repeatable_bitwise():
    w, C = FWD_CASES[0]
    inp = Inputs(w)
    s = inp.shape
    ws = B.workspace(B.expert_choice_workspace_size(s, C))
    a, b = new((w.T, w.d), w.dtype), new((w.T, w.d), w.dtype)
    for o in (a, b):
        B.forward_expert_choice(s, C, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, o, ws)
    assert B.get_error() == B.MOE_OK
    assert torch.equal(a, b)


def test_forward_expert_choice_worked_example_shapes():
    """The worked example's shapes (8192 tokens, d 4096, 64 tanh-GELU experts
    of 16384) with C = T*2/64 = 256 tokens per expert (the compute of top-2):
    the choice checked on every expert, outputs of sampled tokens against the
    oracle."""
    w = S.WORKLOADS["worked-example-n64-f16384-gelu"]
    C = w.T * w.k // w.N
    inp = Inputs(w, host_weights=False)
    s = inp.shape
    g = gpu_route_ec(inp, C)
    check_definition(g, w.T, w.N, C)
    orc = oracle.route(inp.x_h, inp.wg_h, 1, bias=inp.bias_h, want_probs=True)
    check_against_oracle(g, orc["probs"], C)
    out = new((w.T, w.d), w.dtype)
    ws = B.workspace(B.expert_choice_workspace_size(s, C))
    B.forward_expert_choice(s, C, inp.x, inp.wg, inp.bias, inp.w_gate, inp.w_up, inp.w_down, out, ws)
    assert B.get_error() == B.MOE_OK
    picked = np.nonzero(np.any(g["inv"] >= 0, axis=1))[0]
    tokens = np.sort(np.random.default_rng(3).choice(picked, size=16, replace=False))
    ref = ec_reference(inp, g, tokens)
    got = host_f64(out[torch.from_numpy(tokens).cuda()])
    assert rel_err(got, ref) <= tol(w.dtype)


def test_route_expert_choice_empty_batch():
    s = B.shape(0, 128, 8, 2, 64, "swiglu", "bf16")
    counts, offsets = new((8,), "i32", fill=-1), new((9,), "i32", fill=-1)
    wg = torch.zeros((128, 8), dtype=torch.float32, device="cuda")
    B.route_expert_choice(s, 0, None, wg, None, None, None, counts, offsets, None, None)
    assert B.get_error() == B.MOE_OK
    assert counts.cpu().tolist() == [0] * 8 and offsets.cpu().tolist() == [0] * 9


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gather_rows_matches_indexing(dtype):
    """moe_gather_rows with expert-choice tables: row r of x_perm is x[perm[r]];
    slots marked -2 are skipped."""
    w, C = ROUTE_CASES[1][0], 31
    if dtype == "f32":
        w = S.Workload("ec-gather-f32", T=500, d=64, N=16, k=2, F=64, act="swiglu", dtype="f32", seed=78)
    inp = Inputs(w, host_weights=False)
    g = gpu_route_ec(inp, C)
    rows = w.N * C
    xp = new((rows, w.d), dtype, fill=0)
    B.gather_rows(inp.shape, torch.from_numpy(g["inv"]).cuda(), w.N, rows, inp.x, xp)
    assert B.get_error() == B.MOE_OK
    assert torch.equal(xp, inp.x[torch.from_numpy(g["perm"]).long().cuda()])
