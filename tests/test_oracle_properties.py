"""Property tests of the oracle's grouping, capacity, expert-choice and
statistics functions on random small inputs (hypothesis). Each property is a
fact the definitions fix, checked with plain numpy, not a retyped loop of the
oracle: counts are histograms, kept assignments are the earliest ones per
expert, permutations invert each other, expert choice takes each expert's
largest values, fractions sum to one."""
import numpy as np
import pytest
from hypothesis import given, settings, strategies as st

import oracle

SETTINGS = settings(max_examples=60, deadline=None)


@st.composite
def routings(draw):
    N = draw(st.integers(1, 12))
    k = draw(st.integers(1, N))
    T = draw(st.integers(0, 40))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(N, k, replace=False) for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, k), np.int32)
    return idx, N


@SETTINGS
@given(routings(), st.integers(0, 50))
def test_capacity_grouping_properties(rt, cap):
    idx, N = rt
    T, k = idx.shape
    r = oracle.permute_capacity(idx, N, cap)
    demand = np.bincount(idx.ravel(), minlength=N)
    np.testing.assert_array_equal(r["counts"], np.minimum(demand, cap))
    np.testing.assert_array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
    assert r["dropped"] == int(np.maximum(demand - cap, 0).sum())
    flat = idx.ravel()
    inv = r["inv_perm"]
    # an assignment is kept iff fewer than cap earlier assignments went to its expert
    for f in range(T * k):
        e = flat[f]
        earlier = int(np.sum(flat[:f] == e))
        if earlier < cap:
            row = inv[f]
            assert r["offsets"][e] + earlier == row and r["perm"][row] == f // k
        else:
            assert inv[f] == -2
    # the kept rows are a bijection onto [0, offsets[N])
    kept = inv[inv >= 0]
    np.testing.assert_array_equal(np.sort(kept), np.arange(r["offsets"][-1]))


@SETTINGS
@given(routings())
def test_plain_grouping_is_capacity_without_drop(rt):
    idx, N = rt
    T, k = idx.shape
    a = oracle.permute(idx, N)
    b = oracle.permute_capacity(idx, N, T * k)
    for key in ("counts", "offsets", "inv_perm"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_array_equal(a["perm"], b["perm"])
    assert b["dropped"] == 0


@SETTINGS
@given(st.integers(1, 30), st.integers(1, 8), st.integers(0, 2 ** 31 - 1), st.data())
def test_expert_choice_properties(T, N, seed, data):
    C = data.draw(st.integers(0, T))
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, N))
    if data.draw(st.booleans()):
        logits = np.round(logits)                    # many exact ties
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    r = oracle.expert_choice(p, C)
    picked = r["inv"] >= 0
    np.testing.assert_array_equal(picked.sum(0), np.full(N, C))       # equal load, by construction
    for e in range(N):
        rows = r["perm"][e * C:(e + 1) * C]
        assert np.all(np.diff(rows) > 0)                                # ascending token order
        if 0 < C < T:
            chosen = p[rows, e]
            rest = np.delete(p[:, e], rows)
            assert chosen.min() >= rest.max()                           # the C largest
            # at the threshold, the lower token ids win
            tied_left = np.setdiff1d(np.nonzero(p[:, e] == chosen.min())[0], rows)
            tied_in = rows[p[rows, e] == chosen.min()]
            if tied_left.size and tied_in.size:
                assert tied_in.max() < tied_left.min()
    np.testing.assert_array_equal(r["w"][picked], p[picked])
    assert np.all(r["w"][~picked] == 0)


@SETTINGS
@given(routings(), st.integers(0, 2 ** 31 - 1))
def test_load_stats_properties(rt, seed):
    idx, N = rt
    T, k = idx.shape
    rng = np.random.default_rng(seed)
    p = rng.random((T, N)) + 1e-3
    p /= p.sum(1, keepdims=True)
    s = oracle.load_stats(p, idx)
    if T == 0:
        assert s["balance"] == 0.0 and s["entropy_bits"] == 0.0 and s["top1"] == 0.0
        return
    assert s["f"].sum() == pytest.approx(1.0, rel=1e-12)
    assert s["P"].sum() == pytest.approx(1.0, rel=1e-12)
    assert 0.0 <= s["entropy_bits"] <= np.log2(N) + 1e-12
    assert 1.0 / N - 1e-12 <= s["top1"] <= 1.0
    # N sum f P lies between N min(P) and N max(P) (f is a probability vector)
    assert N * s["P"].min() - 1e-12 <= s["balance"] <= N * s["P"].max() + 1e-12
