"""Failure detection without a GPU fault: bad inputs and a bounded device wait
that runs out are reported through the error word, and the context stays
usable afterwards."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import Inputs, host_f64, rel_err, run_forward, tol

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    B.selftest_bounded_wait(20_000_000)          # 20 ms on a barrier nothing completes
    assert B.get_error() == B.MOE_ERR_TIMEOUT
    assert B.get_error() == B.MOE_OK
    # the context still runs the layer correctly
    w = S.Workload("after-timeout", T=64, d=128, N=4, k=2, F=128, act="swiglu", dtype="bf16", seed=5)
    inp = Inputs(w)
    out = run_forward(inp)[0]
    WG = np.stack([inp.host[e][0] for e in range(w.N)])
    WU = np.stack([inp.host[e][1] for e in range(w.N)])
    WD = np.stack([inp.host[e][2] for e in range(w.N)])
    ref = oracle.forward(inp.x_h, inp.wg_h, None, WG, WU, WD, w.k, w.act)
    assert rel_err(host_f64(out), ref["out"]) <= tol("bf16")


def test_corrupt_routing_in_forward_is_reported_not_faulted():
    """An out-of-range expert index fed to the staged path: the permute records
    MOE_ERR_CORRUPT and places only the valid assignments (a prefix of the
    rows, which the GEMMs accept), and the combine skips the slot it cannot
    trust. Nothing reads out of bounds."""
    w = S.Workload("corrupt", T=100, d=128, N=8, k=2, F=128, act="swiglu", dtype="bf16", seed=6)
    inp = Inputs(w)
    s = inp.shape
    idx = torch.randint(0, 8, (w.T, w.k), dtype=torch.int32, device="cuda")
    idx[5, 0] = 1000
    tw = torch.full((w.T, w.k), 0.5, device="cuda")
    counts = torch.empty(8, dtype=torch.int32, device="cuda")
    offsets = torch.empty(9, dtype=torch.int32, device="cuda")
    perm = torch.empty(w.A, dtype=torch.int32, device="cuda")
    inv = torch.empty(w.A, dtype=torch.int32, device="cuda")
    xp = torch.zeros(w.A, w.d, dtype=torch.bfloat16, device="cuda")
    yp = torch.zeros(w.A, w.d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(w.T, w.d, dtype=torch.bfloat16, device="cuda")
    ws = B.workspace(max(B.permute_workspace_size(s), B.grouped_ffn_workspace_size(s)))
    B.permute(s, idx, inp.x, counts, offsets, perm, inv, xp, ws)
    B.grouped_ffn(s, xp, offsets, inp.w_gate, inp.w_up, inp.w_down, yp, ws)
    B.combine(s, yp, inv, tw, out)
    assert B.get_error() == B.MOE_ERR_CORRUPT
    assert B.get_error() == B.MOE_OK
