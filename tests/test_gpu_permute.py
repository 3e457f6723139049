"""moe_permute on the GPU: counts, offsets, perm, inv_perm and x_perm are
bit-exact against the oracle's stable counting sort, for the same top-k input."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import dev, new

pytestmark = pytest.mark.gpu


def run_permute(idx_h, x_h, N, dtype):
    T, k = idx_h.shape
    d = x_h.shape[1]
    s = B.shape(T, d, N, k, 64, "swiglu", dtype)
    A = T * k
    counts = new((N,), "i32", fill=-1)
    offsets = new((N + 1,), "i32", fill=-1)
    perm = new((max(A, 1),), "i32", fill=-1)
    inv = new((max(A, 1),), "i32", fill=-1)
    xp = new((max(A, 1), d), dtype)
    ws = B.workspace(B.permute_workspace_size(s))
    B.permute(s, dev(idx_h), dev(x_h) if T else xp, counts, offsets, perm, inv, xp, ws)
    assert B.get_error() == B.MOE_OK
    return (counts.cpu().numpy(), offsets.cpu().numpy(), perm.cpu().numpy()[:A], inv.cpu().numpy()[:A],
            xp[:A].cpu())


def compare(idx_h, x_h, N, dtype):
    c, o, p, i, xp = run_permute(idx_h, x_h, N, dtype)
    ref = oracle.permute(idx_h, N)
    np.testing.assert_array_equal(c, ref["counts"])
    np.testing.assert_array_equal(o, ref["offsets"])
    np.testing.assert_array_equal(p, ref["perm"])
    np.testing.assert_array_equal(i, ref["inv_perm"])
    xd = dev(x_h).cpu() if x_h.shape[0] else None
    if len(p):
        assert torch.equal(xp, xd[torch.from_numpy(ref["perm"]).long()])   # rows copied bit for bit


def random_idx(T, N, k, seed, skew=None):
    rng = np.random.default_rng(seed)
    if skew is None:
        return np.stack([rng.choice(N, k, replace=False) for _ in range(T)]).astype(np.int32)
    p = np.arange(1, N + 1, dtype=np.float64) ** -skew
    p /= p.sum()
    return np.stack([rng.choice(N, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def xs(T, d, dtype, seed=0):
    w = S.Workload("perm-x", T=max(T, 1), d=d, N=1, k=1, F=64, act="swiglu", dtype=dtype, seed=seed)
    return S.x_all(w)[:T]


@pytest.mark.parametrize("T,N,k,d,dtype", [
    (1, 8, 2, 128, "bf16"),
    (100, 8, 2, 256, "bf16"),
    (1023, 64, 8, 128, "bf16"),      # several chunks, ragged tail
    (3000, 7, 3, 128, "bf16"),       # k not a power of two
    (515, 256, 4, 128, "bf16"),
    (64, 8, 2, 128, "f32"),
    (50, 9, 9, 12, "f32"),           # k = N
    (256, 64, 8, 3584, "bf16"),      # exactly one chunk (2048 assignments): the one-launch grouping
    (1024, 16, 2, 128, "bf16"),      # one chunk
    (1025, 16, 2, 128, "bf16"),      # one token more: two chunks
])
def test_permute_random(T, N, k, d, dtype):
    compare(random_idx(T, N, k, T * 7 + N), xs(T, d, dtype, T), N, dtype)


def test_permute_all_on_one_expert_and_empty_experts():
    T, N, k = 5000, 32, 1
    idx = np.full((T, k), 17, np.int32)
    compare(idx, xs(T, 128, "bf16"), N, "bf16")
    idx = random_idx(4097, 16, 2, 3)
    idx[idx == 5] = 6          # expert 5 empty
    idx = np.where(idx % 4 == 0, 12, idx).astype(np.int32)
    for t in range(idx.shape[0]):       # keep the k experts of a token distinct
        if idx[t, 0] == idx[t, 1]:
            idx[t, 1] = 1 if idx[t, 0] != 1 else 2
    compare(idx, xs(4097, 128, "bf16"), 16, "bf16")


def test_permute_skewed_large():
    """Zipf-skewed routing at the skewed workload's size (131072 assignments)."""
    w = S.WORKLOADS["zipf-skew-n128-k8"]
    compare(random_idx(w.T, w.N, w.k, 11, skew=1.2), xs(w.T, w.d, "bf16", 5), w.N, "bf16")


def test_permute_empty_input():
    c, o, p, i, xp = run_permute(np.zeros((0, 2), np.int32), np.zeros((0, 128), np.uint16), 8, "bf16")
    assert c.tolist() == [0] * 8 and o.tolist() == [0] * 9


@pytest.mark.parametrize("T", [300, 3000])     # one chunk (one launch) and several chunks
def test_permute_corrupt_index_recorded(T):
    idx = random_idx(T, 8, 2, 1)
    idx[17, 1] = 8                     # out of range
    T, k = idx.shape
    s = B.shape(T, 128, 8, k, 64, "swiglu", "bf16")
    x = dev(xs(T, 128, "bf16"))
    counts, offsets = new((8,), "i32"), new((9,), "i32")
    perm, inv = new((T * k,), "i32"), new((T * k,), "i32")
    xp = new((T * k, 128), "bf16")
    ws = B.workspace(B.permute_workspace_size(s))
    B.permute(s, dev(idx), x, counts, offsets, perm, inv, xp, ws)
    assert B.get_error() == B.MOE_ERR_CORRUPT
    assert int(offsets[8].item()) == T * k - 1          # the bad assignment is not counted
    assert int(inv[17 * 2 + 1].item()) == -1
    assert B.get_error() == B.MOE_OK                    # the word was cleared
