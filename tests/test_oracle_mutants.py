"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a transposed
operand, a dropped term, a flipped comparison, a wrong constant, an unstable
order, a wrong sign), builds the copy, and runs the pin it should trip: the
same independent checks the pin tests make (numpy / scipy definitions,
closed forms, invariants). The unmodified oracle passes every check, each
mutant fails its own. Mistakes are planted on the CPU only.
"""
import importlib.util
import math
import os
import shutil

import numpy as np
import pytest
from scipy import special

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.join(os.path.dirname(HERE), "oracle")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ------------------------------------------------------------------ checks (each returns True when it passes)
def check_gate_is_matmul(o):
    x, wg = _rand((17, 9), 1), _rand((9, 5), 2)
    r = o.route(x, wg, 2, want_logits=True, gate="fp64")
    return np.allclose(r["logits"], x @ wg, rtol=1e-12, atol=1e-12)


def check_weights_renormalised(o):
    x, wg = _rand((30, 12), 3), _rand((12, 7), 4)
    r = o.route(x, wg, 3, gate="fp64")
    p = special.softmax(x @ wg, axis=1)
    sel = np.take_along_axis(p, r["topk_idx"].astype(np.int64), 1)
    return np.allclose(r["topk_w"], sel / sel.sum(1, keepdims=True), rtol=1e-12)


def check_tie_rule(o):
    x = np.ones((1, 1))
    wg = np.array([[1.0, 2.0, 2.0, 0.5]])                 # experts 1 and 2 tie
    r = o.route(x, wg, 1, gate="fp64")
    return r["topk_idx"][0, 0] == 1


def check_permute_stable(o):
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(6, 2, replace=False) for _ in range(40)]).astype(np.int32)
    r = o.permute(idx, 6)
    flat = idx.ravel()
    want = np.argsort(flat, kind="stable") // 2             # rows grouped by expert, flat order inside
    return np.array_equal(r["perm"], want)


def check_silu(o):
    v = np.linspace(-4, 4, 9)
    x = np.eye(9)
    W_gate = np.diag(v)
    W_up = np.eye(9)
    y = o.expert_rows(x, W_gate, W_up, np.eye(9), "swiglu")
    return np.allclose(np.diag(y), v * special.expit(v), rtol=1e-13, atol=1e-15)


def check_gelu_tanh(o):
    v = np.linspace(-3, 3, 7)
    y = o.expert_rows(np.eye(7), np.diag(v), None, np.eye(7), "gelu_tanh")
    ref = 0.5 * v * (1 + np.tanh(math.sqrt(2 / math.pi) * (v + 0.044715 * v ** 3)))
    return np.allclose(np.diag(y), ref, rtol=1e-13, atol=1e-15)


def check_combine_weights(o):
    y = _rand((4, 3), 6)
    inv = np.array([2, 0, 1, 3], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5]])
    out = o.combine(y, inv, w)
    ref = np.stack([0.25 * y[2] + 0.75 * y[0], 0.5 * y[1] + 0.5 * y[3]])
    return np.allclose(out, ref, rtol=1e-14)


def check_capacity_earliest(o):
    idx = np.array([[0], [0], [0], [1]], np.int32)
    r = o.permute_capacity(idx, 2, 2)
    return r["inv_perm"].tolist() == [0, 1, -2, 2] and r["dropped"] == 1


def check_balance_uniform(o):
    N, T = 8, 16
    probs = np.full((T, N), 1.0 / N)
    idx = (np.arange(T) % N).astype(np.int32).reshape(T, 1)
    return abs(o.load_stats(probs, idx)["balance"] - 1.0) < 1e-14


def check_expert_choice_top(o):
    p = np.array([[.6, .4], [.7, .3], [.2, .8], [.5, .5]])
    return o.expert_choice(p, 1)["perm"].tolist() == [1, 2]


CHECKS = [check_gate_is_matmul, check_weights_renormalised, check_tie_rule, check_permute_stable, check_silu,
          check_gelu_tanh, check_combine_weights, check_capacity_earliest, check_balance_uniform,
          check_expert_choice_top]

# (name, text in moe_oracle.c, planted replacement, the check that must fail)
MUTANTS = [
    ("transposed W_g", "rd(wg, wg_dt, (int64_t)i * N + n)", "rd(wg, wg_dt, (int64_t)n * d + i)",
     check_gate_is_matmul),
    ("weights not renormalised", "topk_w[t * k + j] = p[order[j]] / sel;", "topk_w[t * k + j] = p[order[j]];",
     check_weights_renormalised),
    ("ties to the higher id", "if (best < 0 || l[n] > l[best]) best = n;", "if (best < 0 || l[n] >= l[best]) best = n;",
     check_tie_rule),
    ("unstable grouping", "int32_t row = fill[e]++;",
     "int32_t row = offsets[e + 1] - 1 - (fill[e]++ - offsets[e]);", check_permute_stable),
    ("SiLU sign", "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));", check_silu),
    ("GELU constant", "0.044715 * v * v * v", "0.04471 * v * v * v", check_gelu_tanh),
    ("combine drops the gate weight", "out[q * d + o] += w * yr[o];", "out[q * d + o] += yr[o];",
     check_combine_weights),
    ("capacity off by one", "if (r < capacity) {", "if (r <= capacity) {", check_capacity_earliest),
    ("balance without the N factor", "out3[0] = (double)N * bal;", "out3[0] = bal;", check_balance_uniform),
    ("expert choice takes the smallest", "if (x->p > y->p) return -1;", "if (x->p < y->p) return -1;",
     check_expert_choice_top),
]


def load_oracle_copy(tmp_path, name, src_text):
    """A package copy of the oracle with the given C source, built in tmp_path."""
    pkg = tmp_path / name
    pkg.mkdir()
    shutil.copy(os.path.join(ORACLE_DIR, "__init__.py"), pkg / "__init__.py")
    (pkg / "moe_oracle.c").write_text(src_text)
    spec = importlib.util.spec_from_file_location(name, pkg / "__init__.py", submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    return mod


def original_source():
    with open(os.path.join(ORACLE_DIR, "moe_oracle.c")) as f:
        return f.read()


def test_unmodified_copy_passes_every_check(tmp_path):
    o = load_oracle_copy(tmp_path, "oracle_copy", original_source())
    for chk in CHECKS:
        assert chk(o), chk.__name__


@pytest.mark.parametrize("name,old,new,chk", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, chk):
    src = original_source()
    assert src.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    o = load_oracle_copy(tmp_path, "oracle_mutant", src.replace(old, new))
    assert not chk(o), f"planted mistake '{name}' went unnoticed by {chk.__name__}"
