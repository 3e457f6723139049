"""moe_permute_noalloc: the permutation for callers that cannot give the
library device scratch memory (a framework that hands a custom operator only
its inputs and outputs, or code that must not call cudaMalloc mid-forward).

Its scratch is a fixed array inside the library instead of a workspace. The
tests call it through the C ABI twice in a row, on different routings, and
require the same bits as moe_permute (the integer outputs and the copied rows
are exact, so the tolerance is zero), including a shape that needs exactly
the whole array. Collected last on purpose."""
import os
import subprocess
import sys

import pytest
import torch

from mixture_experts_layer_97_b300 import binding as B

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRATCH_INTS = 65536                  # MOE_PERMUTE_NOALLOC_SCRATCH_INTS


def _chunk_entries(T, N, k):
    """Histogram entries the permutation needs: ceil(T / max(1, 2048 // k)) * N."""
    tpc = max(1, 2048 // k)
    return -(-T // tpc) * N


def _routing(T, N, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(N, generator=g)[:k] for _ in range(T)]).to(torch.int32)


def _routing_fast(T, N, k, seed):
    """k distinct experts per token without a Python loop over tokens: a random
    start plus k distinct offsets (a random k-subset of 0..N-1, per token)."""
    g = torch.Generator().manual_seed(seed)
    base = torch.randint(0, N, (T, 1), generator=g)
    step = torch.randperm(N, generator=g)[:k].view(1, k)
    return ((base + step) % N).to(torch.int32)


def _outputs(T, N, k, d):
    A = T * k
    return (torch.full((N,), -1, dtype=torch.int32, device="cuda"),
            torch.full((N + 1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((A,), -1, dtype=torch.int32, device="cuda"),
            torch.full((A,), -1, dtype=torch.int32, device="cuda"),
            torch.zeros((A, d), dtype=torch.bfloat16, device="cuda"))


def _compare_twice(T, N, k, d, make_routing):
    s = B.shape(T, d, N, k, 128, "swiglu", "bf16")
    ws = B.workspace(B.permute_workspace_size(s))
    for call in range(2):                      # the shared scratch keeps the previous call's contents
        idx = make_routing(T, N, k, 1000 * call + T).cuda()
        x = torch.randn(T, d, device="cuda").to(torch.bfloat16)
        ref = _outputs(T, N, k, d)
        B.permute(s, idx, x, *ref, ws)
        got = _outputs(T, N, k, d)
        B.permute_noalloc(s, idx, x, *got)
        assert B.get_error() == B.MOE_OK
        for a, b in zip(got, ref):
            assert torch.equal(a, b)
        assert int(got[1][-1].item()) == T * k


@pytest.mark.parametrize("T,N,k,d", [(3000, 64, 2, 256), (777, 128, 8, 128)])
def test_noalloc_permute_matches_workspace_permute_twice(T, N, k, d):
    _compare_twice(T, N, k, d, _routing)


def test_noalloc_permute_at_the_scratch_limit():
    # 65536 tokens, top-8 of 256: 256 tokens per chunk, 256 chunks x 256 experts = every entry of the array
    T, N, k, d = 65536, 256, 8, 128
    assert _chunk_entries(T, N, k) == SCRATCH_INTS
    _compare_twice(T, N, k, d, _routing_fast)


@pytest.mark.parametrize("T,N,k", [(65537, 256, 8), (600_000, 256, 1)])
def test_noalloc_rejects_shapes_beyond_its_scratch(T, N, k):
    """Real device buffers sized for the shape: if the size check ever let the
    call through, the kernels would still run in bounds and the wrong status
    would fail the assert."""
    d = 128
    assert _chunk_entries(T, N, k) > SCRATCH_INTS
    s = B.shape(T, d, N, k, 128, "swiglu", "bf16")
    idx = _routing_fast(T, N, k, 5).cuda()
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    out = _outputs(T, N, k, d)
    with pytest.raises(B.MoEError) as e:
        B.permute_noalloc(s, idx, x, *out)
    assert e.value.status == B.MOE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert B.get_error() == B.MOE_OK
    assert int(out[0][0].item()) == -1               # nothing was launched


_FIRST_USE_FROM_THREADS = r"""
import sys, threading, torch
sys.path.insert(0, sys.argv[1])
from mixture_experts_layer_97_b300 import binding as B
torch.cuda.set_device(0)
T, N, k, d, F = 500, 32, 2, 128, 128
s = B.shape(T, d, N, k, F, "swiglu", "bf16")
idx = torch.stack([torch.randperm(N)[:k] for _ in range(T)]).to(torch.int32).cuda()
x = (torch.randn(T, d, device="cuda")).to(torch.bfloat16)
wg = torch.randn(d, N, device="cuda") * 0.02
W = [torch.randn(N, F, d, device="cuda").mul_(0.02).to(torch.bfloat16) for _ in range(2)]
WD = torch.randn(N, d, F, device="cuda").mul_(0.02).to(torch.bfloat16)
A = T * k
perm_out = (torch.empty(N, dtype=torch.int32, device="cuda"), torch.empty(N + 1, dtype=torch.int32, device="cuda"),
            torch.empty(A, dtype=torch.int32, device="cuda"), torch.empty(A, dtype=torch.int32, device="cuda"),
            torch.empty(A, d, dtype=torch.bfloat16, device="cuda"))
fwd_out = [torch.empty(T, d, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
fwd_ws = [B.workspace(B.workspace_size(s)) for _ in range(2)]
torch.cuda.synchronize()
streams = [torch.cuda.Stream() for _ in range(3)]
errors = []
go = threading.Barrier(3)
def work(i):
    # first library calls of the process, made by three host threads at once: the grouping without a
    # workspace (scratch-address lookup) and two forwards (SM count, tensor-map encoder); the two forwards
    # have their own workspaces and only one call uses the shared scratch array
    try:
        torch.cuda.set_device(0)
        go.wait()
        with torch.cuda.stream(streams[i]):
            if i == 0:
                B.permute_noalloc(s, idx, x, *perm_out)
            else:
                B.forward(s, x, wg, None, W[0], W[1], WD, fwd_out[i - 1], fwd_ws[i - 1])
            streams[i].synchronize()
    except Exception as e:
        errors.append(repr(e))
ts = [threading.Thread(target=work, args=(i,)) for i in range(3)]
for t in ts: t.start()
for t in ts: t.join()
assert not errors, errors
assert B.get_error() == B.MOE_OK
ref = tuple(torch.empty_like(t) for t in perm_out)
B.permute(s, idx, x, *ref, B.workspace(B.permute_workspace_size(s)))
out1 = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
B.forward(s, x, wg, None, W[0], W[1], WD, out1, B.workspace(B.workspace_size(s)))
torch.cuda.synchronize()
for a, b in zip(perm_out, ref):
    assert torch.equal(a, b)
for o in fwd_out:
    assert torch.equal(o, out1)
print("ok")
"""


def test_first_library_calls_from_three_threads_in_a_fresh_process():
    """The first calls in a process fill the library's per-process caches (the
    scratch address, the SM count, the tensor-map encoder): make them from
    three host threads at once in a fresh process and check every result."""
    r = subprocess.run([sys.executable, "-c", _FIRST_USE_FROM_THREADS, ROOT], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
