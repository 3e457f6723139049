"""moe_route on the GPU against the oracle: bit-exact top-k indices on every
token (both sides decide on fp32 logits, the pages' gate precision), weights
within 1e-5, exact ties broken by the lower expert id."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import check_route, dev, new

pytestmark = pytest.mark.gpu


def run_route(x_h, wg_h, bias_h, k, dtype):
    T, d = x_h.shape
    N = wg_h.shape[1]
    s = B.shape(T, d, N, k, 64, "swiglu", dtype)
    idx = new((T, k), "i32", fill=-7)
    w = new((T, k), "f32", fill=-1.0)
    B.route(s, dev(x_h), dev(wg_h), dev(bias_h) if bias_h is not None else None, idx, w)
    assert B.get_error() == B.MOE_OK
    return idx.cpu().numpy(), w.cpu().numpy().astype(np.float64)


CASES = [
    # T, d, N, k, dtype, bias
    (64, 128, 8, 2, "f32", False),
    (1, 128, 8, 2, "bf16", False),
    (65, 256, 16, 1, "bf16", True),
    (200, 384, 17, 3, "bf16", False),
    (257, 128, 64, 8, "bf16", True),
    (130, 512, 128, 8, "bf16", True),
    (96, 256, 256, 16, "bf16", False),
    (33, 256, 8, 8, "bf16", False),       # k = N
    (70, 100, 5, 5, "f32", True),         # d not a multiple of the K slice, N < 16
    (40, 36, 256, 255, "f32", False),
    # token tile per CTA: 4 (small batches), 8, 32, 64 (and 32/64/128 with <= 8 experts)
    (10000, 256, 256, 8, "bf16", True),
    (12000, 64, 5, 2, "f32", False),       # N % 4 != 0: 4-byte copies of W_g
    (5000, 128, 17, 3, "bf16", False),
    (6000, 512, 64, 2, "f32", True),
    (1000, 256, 64, 4, "bf16", False),     # 8 tokens per CTA
    (20000, 128, 8, 2, "bf16", True),      # 8 expert lanes, 128 tokens per CTA
    # the small-batch kernel (64 or 128 experts, one CTA per token, whole-row W_g slices)
    (1, 128, 64, 8, "bf16", False),
    (31, 3584, 64, 8, "bf16", True),
    (300, 384, 128, 8, "bf16", True),
    (17, 256, 64, 2, "f32", True),
    (600, 128, 64, 4, "bf16", False),      # past four CTAs per SM: the generic kernel again
    (8192, 4096, 64, 2, "bf16", False),    # 56 tokens per CTA, 7 per thread
    (16384, 512, 128, 8, "bf16", True),    # 112 tokens per CTA, 7 per thread
]


@pytest.mark.parametrize("T,d,N,k,dtype,use_bias", CASES)
def test_route_matches_oracle(T, d, N, k, dtype, use_bias):
    w = S.Workload("route-case", T=T, d=d, N=N, k=k, F=64, act="swiglu", dtype=dtype, seed=T + d + N + k,
                   zipf_s=1.2 if use_bias else None)
    x_h, wg_h, b_h = S.x_all(w), S.gate_weight(w), S.gate_bias(w)
    gi, gw = run_route(x_h, wg_h, b_h, k, dtype)
    check_route(gi, gw, oracle.route(x_h, wg_h, k, bias=b_h))


def test_route_exact_ties_lower_id_wins():
    """Integer-valued x and W_g (multiples of 1/8): every fp32 sum is exact, so
    ties are real and the rule (lower expert id first) is checked bit-exactly."""
    rng = np.random.default_rng(7)
    T, d, N, k = 300, 128, 16, 4
    x = rng.integers(-2, 3, size=(T, d)).astype(np.float32)
    wg = (rng.integers(-2, 3, size=(d, N)) / 8.0).astype(np.float32)
    wg[:, 5] = wg[:, 3]          # experts 3 and 5 always tie
    wg[:, 9] = wg[:, 2]          # and 2 and 9
    xb = S.f32_to_bf16_bits(x)   # exact in bf16
    gi, gw = run_route(xb, wg, None, k, "bf16")
    orc = oracle.route(xb, wg, k)
    np.testing.assert_array_equal(gi, orc["topk_idx"])
    np.testing.assert_allclose(gw, orc["topk_w"], atol=1e-6)
    L = x.astype(np.float64) @ wg.astype(np.float64)
    ties = np.sum([len(np.unique(L[t])) < N for t in range(T)])
    assert ties > T // 2


@pytest.mark.parametrize("name", ["prefill-n8-f14336", "worked-example-n64-f16384-gelu",
                                  "decode-t32-n64-k8", "zipf-skew-n128-k8"])
def test_route_full_size(name):
    w = S.WORKLOADS[name]
    x_h, wg_h, b_h = S.x_all(w), S.gate_weight(w), S.gate_bias(w)
    gi, gw = run_route(x_h, wg_h, b_h, w.k, w.dtype)
    fragile = check_route(gi, gw, oracle.route(x_h, wg_h, w.k, bias=b_h))
    print(f"{name}: routing bit-exact on all {w.T} tokens ({fragile} with rounding-fragile decisions)")


def test_route_repeatable():
    w = S.WORKLOADS["zipf-skew-n128-k8"].scaled(T=1000)
    x_h, wg_h, b_h = S.x_all(w), S.gate_weight(w), S.gate_bias(w)
    a = run_route(x_h, wg_h, b_h, w.k, w.dtype)
    b = run_route(x_h, wg_h, b_h, w.k, w.dtype)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("T,d,N,k,dtype,mode", [(1, 128, 64, 8, "bf16", "logits"), (40, 3584, 64, 8, "bf16", "select"),
                                                (100, 256, 128, 8, "f32", "logits"),
                                                (7, 1024, 128, 4, "bf16", "select")])
def test_small_batch_kernel_equals_the_generic_kernel(T, d, N, k, dtype, mode):
    """Asking for routing statistics takes the generic kernel; without them a
    small batch takes the small-batch kernel. Both evaluate the same fp32
    chains, so indices and weights agree bit for bit."""
    w = S.Workload("route-small", T=T, d=d, N=N, k=k, F=64, act="swiglu", dtype=dtype, seed=T + d, zipf_s=1.2)
    x_h, wg_h, b_h = S.x_all(w), S.gate_weight(w), S.gate_bias(w)
    s = B.shape(T, d, N, k, 64, "swiglu", dtype)
    x, wg, b = dev(x_h), dev(wg_h), dev(b_h)
    outs = []
    for stats in (False, True):
        idx = new((T, k), "i32", fill=-7)
        tw = new((T, k), "f32", fill=-1.0)
        st = torch.empty(B.load_stats_len(N), dtype=torch.float32, device="cuda") if stats else None
        ws = B.workspace(B.route_ex_workspace_size(s)) if stats else None
        B.route_ex(s, x, wg, b, idx, tw, bias_mode=mode, load_stats=st, ws=ws)
        assert B.get_error() == B.MOE_OK
        outs.append((idx.cpu(), tw.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    r = oracle.route(x_h, wg_h, k, bias=b_h, bias_mode=mode)
    np.testing.assert_array_equal(outs[0][0].numpy(), r["topk_idx"])
