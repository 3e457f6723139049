"""FLOP and byte accounting pinned to the figures printed on the pages
(tests/golden/pages_figures.json, each entry with its citation)."""
import json
import os

import pytest

from mixture_experts_layer_97_b300 import accounting as acc

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


def test_swiglu_flops_match_printed_estimate():
    g = GOLD["flop_estimate"]
    d, F, N, k, S = g["d"], g["d_ff"], g["experts"], g["top_k"], g["tokens"]
    assert 2 * d * F == pytest.approx(g["per_projection_flops_approx"], rel=0.01)
    assert acc.ffn_flops_per_assignment(d, F, "swiglu") == pytest.approx(g["per_token_expert_flops_approx"], rel=0.01)
    assert acc.ffn_flops(k, d, F, "swiglu") == pytest.approx(g["per_token_flops_approx"], rel=0.01)
    assert acc.ffn_flops(S * k, d, F, "swiglu") == pytest.approx(g["layer_flops_approx"], rel=0.02)
    assert acc.ffn_flops(S * N, d, F, "swiglu") == pytest.approx(g["dense_equivalent_flops_approx"], rel=0.02)
    # the split into the two grouped GEMMs adds up
    A = S * k
    assert acc.up_flops(A, d, F, "swiglu") + acc.down_flops(A, d, F) == acc.ffn_flops(A, d, F, "swiglu")


def test_worked_example_weight_bytes():
    g = GOLD["worked_example"]
    one = acc.expert_weight_bytes(g["hidden"], g["ffn_hidden"], "gelu_tanh", 2)
    assert one == pytest.approx(g["expert_bytes_fp16_approx"], rel=0.01)
    assert g["experts"] * one == pytest.approx(g["all_experts_bytes_fp16_approx"], rel=0.02)
    assert acc.active_expert_weight_bytes([1] * 64, g["hidden"], g["ffn_hidden"], "gelu_tanh", 2) == 64 * one
    assert acc.active_expert_weight_bytes([0, 3, 0], 8, 16, "swiglu", 2) == 3 * 8 * 16 * 2


def test_worked_example_output_bytes_corrected():
    g = GOLD["worked_example"]
    T = g["batch"] * g["seq"]
    assert T * g["hidden"] * 2 == g["output_bytes_fp16_correct"]
    assert g["output_bytes_fp16_printed"] == 4 * g["output_bytes_fp16_correct"]


def test_dense_ffn_params():
    g = GOLD["dense_ffn_params"]
    assert acc.expert_weight_bytes(g["hidden"], g["ffn_hidden"], "gelu_tanh", 1) == pytest.approx(
        g["params_approx"], rel=0.05)
