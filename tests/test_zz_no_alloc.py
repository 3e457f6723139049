"""moe_permute_noalloc: the permutation for callers that cannot give the
library device scratch memory (a framework that hands a custom operator only
its inputs and outputs, or code that must not call cudaMalloc mid-forward).

Its scratch is a fixed array inside the library instead of a workspace. The
test calls it through the C ABI twice in a row, on different routings, and
requires the same bits as moe_permute (the integer outputs and the copied
rows are exact, so the tolerance is zero). Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_97_b300 import binding as B

pytestmark = pytest.mark.gpu


def _routing(T, N, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(N, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def _outputs(T, N, k, d):
    A = T * k
    return (torch.full((N,), -1, dtype=torch.int32, device="cuda"),
            torch.full((N + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((A,), -1, dtype=torch.int32, device="cuda"),
            torch.full((A,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros((A, d), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("T,N,k,d", [(3000, 64, 2, 256), (777, 128, 8, 128)])
def test_noalloc_permute_matches_workspace_permute_twice(T, N, k, d):
    s = B.shape(T, d, N, k, 128, "swiglu", "bf16")
    ws = B.workspace(B.permute_workspace_size(s))
    for call in range(2):                      # the shared scratch keeps the previous call's contents
        idx = _routing(T, N, k, 1000 * call + T).cuda()
        x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
        ref = _outputs(T, N, k, d)
        B.permute(s, idx, x, *ref, ws)
        got = _outputs(T, N, k, d)
        B.permute_noalloc(s, idx, x, *got)
        assert B.get_error() == B.MOE_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert int(got[1][-1].item()) == T * k


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # ceil(T / 2048) * 256 chunk-histogram entries exceed the fixed 65536
    s = B.shape(600_000, 128, 256, 1, 128, "swiglu", "bf16")
    p = ctypes.c_void_p(1 << 20)
    st = B.lib().moe_permute_noalloc(ctypes.byref(s), p, p, p, p, p, p, p, None)
    assert st == B.MOE_ERR_WORKSPACE
