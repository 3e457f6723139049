"""Pins of the CPU fp64 oracle against things the pages and mathematics fix.

None of these re-types the oracle's loops: each check is an invariant the pages
state, a closed form, a brute-force enumeration on tiny inputs, a library
routine the step reduces to (matmul, stable sort, softmax, bincount), or a
figure printed on the pages. A plausible slip in the oracle (a transposed
weight, a missing renormalisation, a wrong tie rule, an unstable permutation,
a wrong activation) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy import special

import oracle
from moe_synth import f32_to_bf16_bits, bf16_bits_to_f32

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "pages_figures.json")))


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- gate / route
def test_gate_logits_equal_matmul():
    """logits = x @ W_g (+ b): the pages' gate projection is a plain matmul."""
    x = _rand((37, 24), 1)
    wg = _rand((24, 7), 2, 0.3)
    b = _rand((7,), 3)
    r = oracle.route(x, wg, 3, bias=b, want_logits=True, gate="fp64")
    ref = x @ wg + b
    np.testing.assert_allclose(r["logits"], ref, rtol=1e-12, atol=1e-12)
    # and the transpose would differ: guards the [d, N] layout reading
    assert not np.allclose(r["logits"][:, :7], (x[:, :7] @ wg[:7, :7].T) + b)


def test_gate_reads_fp32_and_bf16_inputs_exactly():
    x32 = _rand((5, 16), 4).astype(np.float32)
    xb = f32_to_bf16_bits(x32)
    wg = _rand((16, 4), 5, 0.1).astype(np.float32)
    r32 = oracle.route(x32, wg, 2, want_logits=True, gate="fp64")
    rb = oracle.route(xb, wg, 2, want_logits=True, gate="fp64")
    np.testing.assert_allclose(r32["logits"], x32.astype(np.float64) @ wg.astype(np.float64), rtol=1e-13)
    np.testing.assert_allclose(rb["logits"],
                               bf16_bits_to_f32(xb).astype(np.float64) @ wg.astype(np.float64), rtol=1e-13)


@pytest.mark.parametrize("N,k", [(5, 1), (5, 2), (6, 3), (7, 4), (6, 6)])
def test_topk_is_bruteforce_best_subset(N, k):
    """Top-k = the k-subset with the largest total score (brute force over all
    subsets), listed in descending score order."""
    T, d = 40, 9
    x = _rand((T, d), 10 + N)
    wg = _rand((d, N), 20 + k)
    b = _rand((N,), 30)
    r = oracle.route(x, wg, k, bias=b, gate="fp64")
    L = x @ wg + b
    for t in range(T):
        best = max(itertools.combinations(range(N), k), key=lambda s: sum(L[t, list(s)]))
        got = r["topk_idx"][t]
        assert sorted(got.tolist()) == sorted(best)
        assert all(L[t, got[j]] > L[t, got[j + 1]] for j in range(k - 1))


def test_topk_tie_rule_lower_id_wins():
    """Exact ties (integer data): the lower expert id is selected and listed first."""
    x = np.array([[1.0]])
    wg = np.array([[2.0, 5.0, 5.0, 1.0, 5.0]])
    r = oracle.route(x, wg, 1)
    assert r["topk_idx"].tolist() == [[1]]
    r = oracle.route(x, wg, 2)
    assert r["topk_idx"].tolist() == [[1, 2]]
    r = oracle.route(x, wg, 4)
    assert r["topk_idx"].tolist() == [[1, 2, 4, 0]]
    np.testing.assert_allclose(r["topk_w"].sum(), 1.0, rtol=1e-15)
    # a tie is never certified
    assert r["cert"][0] <= 0


def test_renormalised_weights_sum_to_one_and_follow_softmax_ratios():
    """g_i' = g_i / sum_sel g: weights sum to 1, and w_a / w_b = p_a / p_b =
    exp(l_a - l_b) because the softmax is proportional to exp(logit)."""
    x = _rand((64, 12), 40)
    wg = _rand((12, 9), 41)
    for k in (1, 2, 3, 5, 9):
        r = oracle.route(x, wg, k, want_logits=True)
        w, idx, L = r["topk_w"], r["topk_idx"], r["logits"]
        np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
        if k == 1:
            np.testing.assert_allclose(w, 1.0, atol=1e-15)
        for t in range(0, 64, 7):
            for a, b in itertools.combinations(range(k), 2):
                np.testing.assert_allclose(w[t, a] / w[t, b], math.exp(L[t, idx[t, a]] - L[t, idx[t, b]]),
                                           rtol=1e-12)


def test_k_equals_n_weights_are_the_full_softmax():
    """With k = N nothing is dropped, so the renormalised weights are the
    softmax over all experts (scipy's softmax as the library routine)."""
    x = _rand((20, 8), 50)
    wg = _rand((8, 6), 51)
    b = _rand((6,), 52)
    r = oracle.route(x, wg, 6, bias=b, gate="fp64")
    P = special.softmax(x @ wg + b, axis=1)
    for t in range(20):
        np.testing.assert_allclose(r["topk_w"][t], P[t, r["topk_idx"][t]], rtol=1e-12)


def test_token_A_printed_example():
    """Token A on experts 0 and 3 with probabilities 0.7 / 0.3 combines as
    0.7 * E0 + 0.3 * E3 (pages' printed example). Build logits ln 0.7, ln 0.3
    with the other experts far below, d = F = 1 experts with closed forms."""
    g = GOLD["worked_example"]["token_A"]
    x = np.array([[1.0]])
    wg = np.array([[math.log(0.7), -40.0, -40.0, math.log(0.3)]])
    r = oracle.route(x, wg, 2, gate="fp64")
    assert r["topk_idx"].tolist() == [g["experts"]]
    np.testing.assert_allclose(r["topk_w"][0], g["probs"], rtol=1e-12)
    # SwiGLU experts with d = F = 1: y = c * silu(a x) * (b x)
    a = np.array([0.5, 1.0, -1.0, 2.0]); bb = np.array([1.5, 1.0, 1.0, -0.5]); c = np.array([2.0, 1.0, 1.0, 3.0])
    WG = a.reshape(4, 1, 1); WU = bb.reshape(4, 1, 1); WD = c.reshape(4, 1, 1)
    f = oracle.forward(x, wg, None, WG, WU, WD, 2, "swiglu", gate="fp64")
    def E(e):
        v = a[e]
        return c[e] * (v / (1 + math.exp(-v))) * bb[e]
    np.testing.assert_allclose(f["out"][0, 0], 0.7 * E(0) + 0.3 * E(3), rtol=1e-12)


def test_error_bound_covers_fp32_evaluations():
    """errb bounds |fl32(l) - l| for any summation order: check against fp32
    sums taken sequentially, reversed, pairwise (numpy) and with a bias add."""
    rng = np.random.default_rng(60)
    T, d, N = 16, 512, 8
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (0.02 * rng.standard_normal((d, N))).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    r = oracle.route(x, wg, 2, bias=b, want_logits=True, gate="fp64")
    r32 = oracle.route(x, wg, 2, bias=b, want_logits=True)
    prods = x[:, :, None] * wg[None, :, :]               # fp32 products [T, d, N]
    seq = np.zeros((T, N), np.float32)
    for i in range(d):
        seq = seq + prods[:, i, :]
    rev = np.zeros((T, N), np.float32)
    for i in reversed(range(d)):
        rev = rev + prods[:, i, :]
    pair = prods.sum(axis=1, dtype=np.float32)
    for s32 in (seq, rev, pair):
        l32 = (s32 + b).astype(np.float64)
        assert np.all(np.abs(l32 - r["logits"]) <= r["errb"])
    assert np.all(np.abs(r32["logits"] - r["logits"]) <= r["errb"])
    assert np.all(r["errb"] > 0)
    # the bound is not vacuous: within ~1e3 ulps of the logit scale
    assert np.all(r["errb"] < 1e-3)


def test_cert_positive_on_continuous_data():
    x = _rand((200, 64), 70).astype(np.float32)
    wg = (0.02 * _rand((64, 16), 71)).astype(np.float32)
    r = oracle.route(x, wg, 4)
    assert (r["cert"] > 0).mean() > 0.95
    # a bias with gaps of 10 separates the experts: the certificate (about the
    # exact logits, bias included) is close to the gap
    b = (10.0 * np.arange(16)).astype(np.float32)
    r = oracle.route(0.01 * x, wg, 4, bias=b)
    assert np.all(r["cert"] > 9.0)
    assert r["topk_idx"].tolist() == [[15, 14, 13, 12]] * 200


# ---------------------------------------------------------------- permutation
def _random_routing(T, N, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.choice(N, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,N,k", [(1, 1, 1), (33, 5, 2), (100, 8, 8), (257, 16, 3)])
def test_permute_matches_stable_sort(T, N, k):
    """counts = bincount, offsets = cumsum with offsets[N] = T*k (the pages'
    sum N_i = B*S*k), rows = a stable sort of the flat assignments by expert."""
    idx = _random_routing(T, N, k, T + N)
    p = oracle.permute(idx, N)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(p["counts"], np.bincount(flat, minlength=N))
    assert p["counts"].sum() == T * k
    np.testing.assert_array_equal(p["offsets"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=N))]))
    order = np.argsort(flat, kind="stable")            # row -> flat assignment
    np.testing.assert_array_equal(p["perm"], order // k)
    inv = np.empty_like(order)
    inv[order] = np.arange(T * k)
    np.testing.assert_array_equal(p["inv_perm"], inv)
    # bijection and round trip
    assert sorted(p["inv_perm"].tolist()) == list(range(T * k))
    np.testing.assert_array_equal(p["perm"][p["inv_perm"]], np.arange(T * k) // k)


def test_permute_empty_experts_and_all_on_one():
    idx = np.full((10, 1), 3, np.int32)
    p = oracle.permute(idx, 6)
    assert p["counts"].tolist() == [0, 0, 0, 10, 0, 0]
    assert p["offsets"].tolist() == [0, 0, 0, 0, 10, 10, 10]
    assert p["perm"].tolist() == list(range(10))


def test_permute_rejects_bad_index():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 7]], np.int32), 4)


def test_worked_example_assignment_total():
    """[4, 2048] tokens, 64 experts, top-2: the N_i sum to 16,384 and the
    top-k tensors have 16,384 elements (printed)."""
    g = GOLD["worked_example"]
    T = g["batch"] * g["seq"]
    idx = _random_routing(T, g["experts"], g["top_k"], 80)
    p = oracle.permute(idx, g["experts"])
    assert int(p["counts"].sum()) == g["assignments_total"] == idx.size == g["topk_elements"]
    assert T * g["experts"] == g["logits_elements"]
    assert g["logits_elements"] * 2 == g["logits_bytes_fp16"]
    assert g["topk_elements"] * (4 + 2) == g["topk_bytes_int32_plus_fp16"]


# ---------------------------------------------------------------- expert FFN
def test_activation_closed_forms():
    """d = F = 1 experts: SwiGLU y = c * silu(a x) * (b x) with silu(v) =
    v * sigmoid(v) (scipy's expit); GELU y = c * gelu_tanh(a x) with the
    textbook tanh form; both checked at several points."""
    for xv in (-3.0, -0.7, 0.0, 0.4, 2.5):
        x = np.array([[xv]])
        a, b, c = 0.9, -1.3, 1.7
        y = oracle.expert_rows(x, np.array([[a]]), np.array([[b]]), np.array([[c]]), "swiglu")
        v = a * xv
        np.testing.assert_allclose(y[0, 0], c * v * special.expit(v) * (b * xv), rtol=1e-13, atol=1e-300)
        y = oracle.expert_rows(x, np.array([[a]]), None, np.array([[c]]), "gelu_tanh")
        ref = c * 0.5 * v * (1 + math.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
        np.testing.assert_allclose(y[0, 0], ref, rtol=1e-13, atol=1e-300)


def test_gelu_tanh_is_close_to_exact_gelu():
    """The tanh form approximates GELU(v) = v * Phi(v) (scipy's ndtr) to a few
    1e-4: pins that the oracle uses a GELU, not another activation."""
    v = np.linspace(-6, 6, 241)
    y = np.array([oracle.expert_rows(np.array([[t]]), np.array([[1.0]]), None, np.array([[1.0]]),
                                     "gelu_tanh")[0, 0] for t in v])
    assert np.max(np.abs(y - v * special.ndtr(v))) < 1e-3
    assert abs(y[np.argmin(np.abs(v - 1.0))] - 0.8411919906082768) < 1e-12


@pytest.mark.parametrize("act", ["swiglu", "gelu_tanh"])
def test_expert_rows_equal_matmul_form(act):
    """Row-by-row loops equal the batched matrix form of the same FFN built
    from library matmuls: y = W_down (act(W_gate X^T) [* W_up X^T])."""
    rng = np.random.default_rng(90)
    n, d, F = 6, 10, 14
    X = rng.standard_normal((n, d))
    Wg = rng.standard_normal((F, d)) * 0.3
    Wu = rng.standard_normal((F, d)) * 0.3 if act == "swiglu" else None
    Wd = rng.standard_normal((d, F)) * 0.3
    y, h = oracle.expert_rows(X, Wg, Wu, Wd, act, want_h=True)
    G = X @ Wg.T
    if act == "swiglu":
        H = G * special.expit(G) * (X @ Wu.T)
    else:
        H = 0.5 * G * (1 + np.tanh(math.sqrt(2 / math.pi) * (G + 0.044715 * G ** 3)))
    np.testing.assert_allclose(h, H, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(y, H @ Wd.T, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("act", ["swiglu", "gelu_tanh"])
def test_identical_experts_give_dense_ffn(act):
    """All experts equal => for any routing the layer is one dense FFN, since
    the renormalised weights sum to 1 (pages: weighted sum of expert outputs)."""
    rng = np.random.default_rng(100)
    T, d, N, k, F = 23, 12, 5, 3, 16
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((d, N))
    Wg1 = rng.standard_normal((F, d)) * 0.2
    Wu1 = rng.standard_normal((F, d)) * 0.2
    Wd1 = rng.standard_normal((d, F)) * 0.2
    WG = np.repeat(Wg1[None], N, 0)
    WU = np.repeat(Wu1[None], N, 0) if act == "swiglu" else None
    WD = np.repeat(Wd1[None], N, 0)
    f = oracle.forward(x, wg, None, WG, WU, WD, k, act, gate="fp64")
    G = x @ Wg1.T
    H = G * special.expit(G) * (x @ Wu1.T) if act == "swiglu" else \
        0.5 * G * (1 + np.tanh(math.sqrt(2 / math.pi) * (G + 0.044715 * G ** 3)))
    np.testing.assert_allclose(f["out"], H @ Wd1.T, rtol=1e-10, atol=1e-12)


def test_k_equals_n_is_the_full_softmax_mixture():
    """k = N: out = sum_n softmax(l)_n * E_n(x), computed without any routing."""
    rng = np.random.default_rng(110)
    T, d, N, F = 9, 8, 4, 6
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((d, N))
    b = rng.standard_normal(N)
    WG = rng.standard_normal((N, F, d)) * 0.3
    WU = rng.standard_normal((N, F, d)) * 0.3
    WD = rng.standard_normal((N, d, F)) * 0.3
    f = oracle.forward(x, wg, b, WG, WU, WD, N, "swiglu", gate="fp64")
    P = special.softmax(x @ wg + b, axis=1)
    ref = np.zeros((T, d))
    for n in range(N):
        G = x @ WG[n].T
        ref += P[:, n:n + 1] * ((G * special.expit(G) * (x @ WU[n].T)) @ WD[n].T)
    np.testing.assert_allclose(f["out"], ref, rtol=1e-10, atol=1e-12)


def test_forward_bruteforce_per_token_loop():
    """Tiny case (2 x 8 tokens, d 16, 4 experts, top-2 -- the shapes of the
    pages' toy forward): each output row equals the per-token definition
    sum_j w_j E_{e_j}(x_t) with experts from library matmuls, and the
    permuted rows hold x of the right token."""
    rng = np.random.default_rng(120)
    T, d, N, k, F = 16, 16, 4, 2, 24
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((d, N)) * 0.5).astype(np.float32)
    WG = rng.standard_normal((N, F, d)) * 0.2
    WU = rng.standard_normal((N, F, d)) * 0.2
    WD = rng.standard_normal((N, d, F)) * 0.2
    f = oracle.forward(x, wg, None, WG, WU, WD, k, "swiglu", gate="fp64")
    L = x.astype(np.float64) @ wg.astype(np.float64)
    for t in range(T):
        sel = sorted(range(N), key=lambda n: (-L[t, n], n))[:k]
        p = special.softmax(L[t])[sel]
        p = p / p.sum()
        ref = np.zeros(d)
        for j, e in enumerate(sel):
            G = WG[e] @ x[t]
            ref += p[j] * (WD[e] @ (G * special.expit(G) * (WU[e] @ x[t])))
        np.testing.assert_allclose(f["out"][t], ref, rtol=1e-10, atol=1e-12)
        for j in range(k):
            assert f["perm"][f["inv_perm"][t * k + j]] == t


def test_forward_is_equivariant_under_token_order():
    """Tokens are independent ("MoE混合专家模型计算原理与推理部署实战解析"
    section 2.2: each token is routed and mixed on its own): reordering the
    batch reorders the output rows the same way and changes no value, while
    the grouping (offsets, counts) only depends on the multiset of choices.
    Catches a combine or permutation that mixes up token and slot indices."""
    rng = np.random.default_rng(121)
    T, d, N, k, F = 23, 16, 6, 3, 20
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (rng.standard_normal((d, N)) * 0.5).astype(np.float32)
    WG = rng.standard_normal((N, F, d)) * 0.2
    WU = rng.standard_normal((N, F, d)) * 0.2
    WD = rng.standard_normal((N, d, F)) * 0.2
    order = rng.permutation(T)
    a = oracle.forward(x, wg, None, WG, WU, WD, k, "swiglu")
    b = oracle.forward(x[order], wg, None, WG, WU, WD, k, "swiglu")
    np.testing.assert_array_equal(b["out"], a["out"][order])
    np.testing.assert_array_equal(b["counts"], a["counts"])


def test_combine_one_hot_and_order():
    y = np.arange(12, dtype=np.float64).reshape(4, 3)
    inv = np.array([2, 0, 3, 1], np.int32)     # T=2, k=2
    w = np.array([[1.0, 0.0], [0.25, 0.75]])
    out = oracle.combine(y, inv, w)
    np.testing.assert_allclose(out[0], y[2])
    np.testing.assert_allclose(out[1], 0.25 * y[3] + 0.75 * y[1])
    out = oracle.combine(y, inv, w, tokens=[1])
    np.testing.assert_allclose(out[0], 0.25 * y[3] + 0.75 * y[1])


# ---------------------------------------------------------------- fp32 gate
def _round_f32(q):
    """Round an exact rational to the nearest fp32, ties to even."""
    from fractions import Fraction
    c0 = np.float32(float(q))
    cands = [c0, np.nextafter(c0, np.float32(np.inf)), np.nextafter(c0, np.float32(-np.inf))]
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - q), int(np.array(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_fp32_gate_is_the_sequential_fma_chain():
    """The pages keep the gate in FP32. The oracle's fp32 logit is, bit for
    bit, s <- fl32(x_i * W_g[i,n] + s) (one rounding per step: an FMA) over
    i = 0..d-1 from 0, then fl32(s + b) -- checked against exact rational
    arithmetic rounded to fp32 by hand."""
    from fractions import Fraction
    rng = np.random.default_rng(130)
    T, d, N = 4, 13, 3
    x = rng.standard_normal((T, d)).astype(np.float32)
    wg = (0.3 * rng.standard_normal((d, N))).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    r = oracle.route(x, wg, 1, bias=b, want_logits=True)
    for t in range(T):
        for n in range(N):
            s = np.float32(0.0)
            for i in range(d):
                s = _round_f32(Fraction(float(x[t, i])) * Fraction(float(wg[i, n])) + Fraction(float(s)))
            s = np.float32(s + b[n])
            assert np.float32(r["logits"][t, n]) == s and float(s) == r["logits"][t, n]


def test_fp32_decisions_differ_from_exact_only_on_uncertified_tokens():
    """Where rounding can change the top-k (cert <= 0) the fp32 and exact
    decisions may differ; everywhere else they must agree."""
    rng = np.random.default_rng(140)
    x = rng.standard_normal((3000, 256)).astype(np.float32)
    wg = (0.02 * rng.standard_normal((256, 64))).astype(np.float32)
    for b in (None, rng.standard_normal(64).astype(np.float32)):
        r32 = oracle.route(x, wg, 4, bias=b)
        r64 = oracle.route(x, wg, 4, bias=b, gate="fp64")
        same = np.all(r32["topk_idx"] == r64["topk_idx"], axis=1)
        assert np.all(same[r64["cert"] > 0])
        assert same.mean() > 0.99
        np.testing.assert_array_equal(r32["cert"], r64["cert"])


# ---------------------------------------------------------------- capacity / token drop
def test_capacity_formula_on_the_worked_example():
    """capacity = capacity_factor * total / num_experts (rounded up), with total
    = T*k assignments: 16384 / 64 = 256 at 1.0, 320 at 1.25."""
    g = GOLD["capacity"]
    T, N, k = 8192, g["worked_example_experts"], 2
    assert T * k == g["worked_example_assignments"]
    assert oracle.capacity(T, N, k, 1.0) == g["capacity_at_1_0"]
    assert oracle.capacity(T, N, k, 1.25) == g["capacity_at_1_25"]
    assert oracle.capacity(10, 3, 1, 1.0) == 4            # ceil(10/3)


@pytest.mark.parametrize("T,N,k,cap", [(40, 5, 2, 10), (200, 8, 3, 50), (97, 16, 4, 1), (30, 4, 2, 0)])
def test_capacity_keeps_the_earliest_assignments(T, N, k, cap):
    """Each expert keeps its first `cap` assignments in flat order (a stable
    sort by expert, then the head of every group); counts = min(demand, cap),
    offsets their cumulative sum, dropped = the rest."""
    rng = np.random.default_rng(T + cap)
    skew = np.arange(1, N + 1, dtype=np.float64) ** -1.5
    idx = np.stack([rng.choice(N, k, replace=False, p=skew / skew.sum()) for _ in range(T)]).astype(np.int32)
    r = oracle.permute_capacity(idx, N, cap)
    flat = idx.reshape(-1)
    demand = np.bincount(flat, minlength=N)
    np.testing.assert_array_equal(r["counts"], np.minimum(demand, cap))
    np.testing.assert_array_equal(r["offsets"], np.concatenate([[0], np.cumsum(np.minimum(demand, cap))]))
    assert r["dropped"] == int(np.maximum(demand - cap, 0).sum())
    assert int(r["counts"].sum()) + r["dropped"] == T * k
    order = np.argsort(flat, kind="stable")                # flat assignments grouped by expert
    group_start = np.concatenate([[0], np.cumsum(demand)])
    kept_rows = []
    for e in range(N):
        kept_rows += list(order[group_start[e]:group_start[e] + min(demand[e], cap)])
    kept_rows = np.array(kept_rows, dtype=np.int64)
    np.testing.assert_array_equal(r["perm"], kept_rows // k)
    inv = np.full(T * k, -2)
    inv[kept_rows] = np.arange(len(kept_rows))
    np.testing.assert_array_equal(r["inv_perm"], inv)


def test_capacity_at_or_above_demand_is_the_plain_grouping():
    idx = _random_routing(150, 6, 2, 5)
    big = oracle.permute_capacity(idx, 6, 10 ** 6)
    plain = oracle.permute(idx, 6)
    assert big["dropped"] == 0
    for key in ("counts", "offsets", "perm", "inv_perm"):
        np.testing.assert_array_equal(big[key], plain[key])


def test_dropped_assignment_adds_nothing_to_the_output():
    """Token A of the pages' example (experts 0 and 3, weights 0.7 / 0.3): if
    expert 3 is over capacity, the layer output is 0.7 * E0(x) alone (no
    renormalisation); with capacity 0 the output is zero."""
    y = np.array([[2.0], [5.0]])                     # rows: E0(x) for token 0, E3(x) for token 0
    w = np.array([[0.7, 0.3]])
    assert oracle.combine(y, np.array([0, -2], np.int32), w)[0, 0] == pytest.approx(0.7 * 2.0)
    assert oracle.combine(y, np.array([-2, -2], np.int32), w)[0, 0] == 0.0
    assert oracle.combine(y, np.array([0, 1], np.int32), w)[0, 0] == pytest.approx(0.7 * 2.0 + 0.3 * 5.0)


# ---------------------------------------------------------------- selection-only bias / load statistics
def _one_hot_gate(logit_rows):
    """x = identity rows, so the logits are exactly the rows of W_g."""
    g = np.asarray(logit_rows, dtype=np.float64)
    return np.eye(g.shape[0]), g


def test_selection_only_bias_hand_case():
    """A bias that flips the choice: logits ln .5, ln .3, ln .2 and bias
    (0, 0, 10), top-2. Both modes choose experts 2 and 0; selection-only
    weights are .2/.7 and .5/.7, bias-in-logits weights come from
    softmax(l + b) restricted to the pair."""
    x, wg = _one_hot_gate([[math.log(.5), math.log(.3), math.log(.2)]])
    b = np.array([0.0, 0.0, 10.0])
    sel = oracle.route(x, wg, 2, bias=b, gate="fp64", bias_mode="select")
    lgt = oracle.route(x, wg, 2, bias=b, gate="fp64", bias_mode="logits")
    assert sel["topk_idx"].tolist() == [[2, 0]] and lgt["topk_idx"].tolist() == [[2, 0]]
    np.testing.assert_allclose(sel["topk_w"][0], [.2 / .7, .5 / .7], rtol=1e-14)
    e10 = math.exp(10.0)
    np.testing.assert_allclose(lgt["topk_w"][0], [.2 * e10 / (.2 * e10 + .5), .5 / (.2 * e10 + .5)], rtol=1e-14)
    assert "4.4" in GOLD["selection_only_bias"]["_cite"]   # the reading pinned here, with its citation


def test_selection_only_bias_matches_its_definition():
    """Selection by argsort of x@W_g + b (stable: lower id first on ties),
    weights = softmax(x@W_g) over the chosen experts, renormalised (matmul,
    stable sort and scipy's softmax as the independent routines)."""
    T, d, N, k = 60, 12, 9, 3
    x = _rand((T, d), 71)
    wg = _rand((d, N), 72, 0.5)
    b = _rand((N,), 73, 2.0)
    r = oracle.route(x, wg, k, bias=b, gate="fp64", bias_mode="select", want_probs=True)
    g = x @ wg
    order = np.argsort(-(g + b), axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(r["topk_idx"], order)
    p = special.softmax(g, axis=1)
    np.testing.assert_allclose(r["probs"], p, rtol=1e-12)
    sel = np.take_along_axis(p, order, 1)
    np.testing.assert_allclose(r["topk_w"], sel / sel.sum(1, keepdims=True), rtol=1e-12)
    # the bias-in-logits mode differs on this input (the pin separates the modes)
    r2 = oracle.route(x, wg, k, bias=b, gate="fp64", bias_mode="logits", want_probs=True)
    np.testing.assert_allclose(r2["probs"], special.softmax(g + b, axis=1), rtol=1e-12)
    assert not np.allclose(r2["topk_w"], r["topk_w"])


def test_selection_only_bias_invariances():
    """Zero bias is the plain route; adding one constant to every expert's
    bias changes nothing in either mode (softmax and the ordering are shift
    invariant)."""
    x = _rand((30, 8), 81)
    wg = _rand((8, 6), 82, 0.5)
    b = _rand((6,), 83)
    plain = oracle.route(x, wg, 2, gate="fp64")
    zero = oracle.route(x, wg, 2, bias=np.zeros(6), gate="fp64", bias_mode="select")
    np.testing.assert_array_equal(zero["topk_idx"], plain["topk_idx"])
    np.testing.assert_allclose(zero["topk_w"], plain["topk_w"], rtol=1e-15)
    for mode in ("select", "logits"):
        a = oracle.route(x, wg, 2, bias=b, gate="fp64", bias_mode=mode)
        c = oracle.route(x, wg, 2, bias=b + 0.25, gate="fp64", bias_mode=mode)
        np.testing.assert_array_equal(a["topk_idx"], c["topk_idx"])
        np.testing.assert_allclose(a["topk_w"], c["topk_w"], rtol=1e-12)


def test_fp32_selection_only_scores_add_the_bias_in_fp32():
    """With the fp32 gate, the choosing score is fl32(fl32 logit + b): equal
    to the bias-in-logits mode's score, so both modes choose the same experts."""
    x = f32_to_bf16_bits(_rand((50, 64), 91).astype(np.float32))
    wg = _rand((64, 16), 92, 0.05).astype(np.float32)
    b = _rand((16,), 93, 0.5).astype(np.float32)
    a = oracle.route(x, wg, 4, bias=b, bias_mode="select", want_logits=True)
    c = oracle.route(x, wg, 4, bias=b, bias_mode="logits", want_logits=True)
    np.testing.assert_array_equal(a["topk_idx"], c["topk_idx"])
    np.testing.assert_array_equal(a["logits"], c["logits"])


def test_balance_quantity_is_one_for_uniform_routing():
    """[P3] s4.2: f_i = P_i = 1/N gives N * sum f_i P_i = 1 (the page's own
    example); the entropy of a uniform load is log2 N and the top-1
    probability is 1/N."""
    for N, k, T in [(4, 1, 8), (8, 2, 12), (16, 4, 20), (64, 2, 64)]:
        probs = np.full((T, N), 1.0 / N)
        idx = np.array([[(t * k + j) % N for j in range(k)] for t in range(T)], np.int32)
        st = oracle.load_stats(probs, idx)
        assert st["balance"] == pytest.approx(GOLD["balance_loss_uniform"]["value"], rel=1e-14)
        assert st["entropy_bits"] == pytest.approx(math.log2(N), rel=1e-14)
        assert st["top1"] == pytest.approx(1.0 / N, rel=1e-14)
        np.testing.assert_allclose(st["f"], 1.0 / N, rtol=1e-14)


def test_activation_entropy_maximum_on_the_page():
    """The page's 16-expert model has a maximum activation entropy of 4.0."""
    g = GOLD["activation_entropy"]
    N = g["experts"]
    probs = np.full((N, N), 1.0 / N)
    idx = np.arange(N, dtype=np.int32).reshape(N, 1)
    assert oracle.load_stats(probs, idx)["entropy_bits"] == pytest.approx(g["max_bits"], abs=1e-14)


def test_balance_quantity_collapse():
    """Every token to expert 0 with probability 1: f_0 = P_0 = 1, so the
    quantity is N; the entropy is 0 and the top-1 probability 1."""
    N, T = 8, 10
    probs = np.zeros((T, N))
    probs[:, 0] = 1.0
    st = oracle.load_stats(probs, np.zeros((T, 1), np.int32))
    assert st["balance"] == N and st["entropy_bits"] == 0.0 and st["top1"] == 1.0


def test_load_stats_against_library_routines():
    """f = bincount / (T k), P = column mean of the softmax (scipy), top1 =
    row max; sum f = sum P = 1; 0 <= entropy <= log2 N."""
    T, d, N, k = 200, 16, 12, 3
    x = _rand((T, d), 101)
    wg = _rand((d, N), 102, 0.4)
    r = oracle.route(x, wg, k, gate="fp64", want_probs=True)
    st = oracle.load_stats(r["probs"], r["topk_idx"])
    f = np.bincount(r["topk_idx"].ravel(), minlength=N) / (T * k)
    p = special.softmax(x @ wg, axis=1)
    np.testing.assert_allclose(st["f"], f, rtol=1e-14)
    np.testing.assert_allclose(st["P"], p.mean(0), rtol=1e-12)
    assert st["top1"] == pytest.approx(p.max(1).mean(), rel=1e-12)
    assert st["f"].sum() == pytest.approx(1.0, rel=1e-14) and st["P"].sum() == pytest.approx(1.0, rel=1e-12)
    assert 0.0 <= st["entropy_bits"] <= math.log2(N)
    assert st["entropy_bits"] == pytest.approx(-(f[f > 0] * np.log2(f[f > 0])).sum(), rel=1e-13)


def test_load_stats_empty_batch():
    st = oracle.load_stats(np.zeros((0, 5)), np.zeros((0, 2), np.int32))
    assert st["balance"] == 0.0 and st["entropy_bits"] == 0.0 and st["top1"] == 0.0


# ---------------------------------------------------------------- expert-choice routing
def _probs(T, N, seed, scale=1.0):
    return special.softmax(_rand((T, N), seed, scale), axis=1)


@pytest.mark.parametrize("T,N,C", [(10, 3, 4), (50, 8, 13), (64, 5, 64), (7, 7, 0), (30, 4, 1)])
def test_expert_choice_matches_lexsort(T, N, C):
    """Each expert's tokens = the first C of a lexicographic sort by (p
    descending, token ascending) -- numpy's lexsort as the independent
    routine; rows list them in ascending token order; every expert gets
    exactly C (the page's balanced load)."""
    p = _probs(T, N, T + N)
    r = oracle.expert_choice(p, C)
    assert r["perm"].shape == (N * C,)
    for e in range(N):
        order = np.lexsort((np.arange(T), -p[:, e]))[:C]
        rows = r["perm"][e * C:(e + 1) * C]
        np.testing.assert_array_equal(rows, np.sort(order))
        np.testing.assert_array_equal(r["w_row"][e * C:(e + 1) * C], p[rows, e])
        if C:
            assert r["thr"][e] == p[order[-1], e]
        assert (r["inv"][:, e] >= 0).sum() == C
    # inv / w are the inverse of perm / w_row
    for row in range(N * C):
        t, e = r["perm"][row], row // C
        assert r["inv"][t, e] == row and r["w"][t, e] == p[t, e]
    assert np.all((r["inv"] >= 0) | (r["inv"] == -2))
    assert np.all(r["w"][r["inv"] == -2] == 0.0)


def test_expert_choice_ties_take_the_lower_token():
    p = np.array([[.5, .5], [.5, .5], [.9, .1], [.5, .5]])
    r = oracle.expert_choice(p, 2)
    assert r["perm"].tolist() == [0, 2, 0, 1]       # expert 0: .9 then the first .5; expert 1: tokens 0, 1


def test_expert_choice_can_leave_a_token_unpicked():
    """[P3] s2.3: a token may be picked by no expert."""
    p = np.array([[.6, .4], [.7, .3], [.2, .8], [.5, .5]])
    r = oracle.expert_choice(p, 1)
    assert r["perm"].tolist() == [1, 2]
    assert np.all(r["inv"][0] == -2) and np.all(r["inv"][3] == -2)
    assert "2.3" in GOLD["expert_choice"]["_cite"]


def test_expert_choice_all_tokens_with_identical_experts_is_the_dense_ffn():
    """C = T: every expert takes every token; with N identical experts the
    combine gives sum_e p[t,e] * FFN(x_t) = FFN(x_t), because the
    probabilities of a token sum to 1 (the dense tanh-GELU FFN is written out
    here with numpy)."""
    T, d, N, F = 12, 16, 4, 24
    x = _rand((T, d), 111)
    wg = _rand((d, N), 112, 0.5)
    W1 = _rand((F, d), 113, 0.3)
    W2 = _rand((d, F), 114, 0.3)
    r = oracle.route(x, wg, 1, gate="fp64", want_probs=True)
    ec = oracle.expert_choice(r["probs"], T)
    y = np.zeros((N * T, d))
    for e in range(N):
        rows = ec["perm"][e * T:(e + 1) * T]
        y[e * T:(e + 1) * T] = oracle.expert_rows(x[rows], W1, None, W2, "gelu_tanh")
    out = oracle.combine(y, ec["inv"], ec["w"])
    hpre = x @ W1.T
    dense = (0.5 * hpre * (1 + np.tanh(np.sqrt(2 / np.pi) * (hpre + 0.044715 * hpre ** 3)))) @ W2.T
    np.testing.assert_allclose(out, dense, rtol=1e-12, atol=1e-12)


def test_expert_choice_rejects_capacity_above_tokens():
    with pytest.raises(ValueError):
        oracle.expert_choice(_probs(4, 2, 1), 5)
