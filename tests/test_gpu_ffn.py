"""moe_grouped_ffn on the GPU against the oracle's per-expert FFN: every row
of y_perm within 2e-2 * max|ref| (bf16, tcgen05 path) or 1e-4 (fp32 path).
Row counts cover empty experts, single rows, exact tile multiples, tile + 1
and ragged tails; shapes cover every kernel variant (SwiGLU 256/128-wide,
GELU 256/128-wide, down 256/128-wide) and more tiles than SMs."""
import numpy as np
import pytest
import torch

import moe_synth as S
import oracle
from mixture_experts_layer_97_b300 import binding as B
from tests.gpu_util import dev, host_f64, new, rel_err, tol

pytestmark = pytest.mark.gpu


def make_case(counts, d, F, act, dtype, seed):
    N = len(counts)
    A = int(sum(counts))
    w = S.Workload("ffn-case", T=A, d=d, N=N, k=1, F=F, act=act, dtype=dtype, seed=seed)
    x_perm = S.x_all(w)                               # rows already grouped by expert
    weights = [S.expert_weights(w, e) for e in range(N)]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return w, x_perm, weights, offsets


def run_ffn(w, x_perm, weights, offsets):
    N, A = w.N, w.T
    s = B.shape(A, w.d, N, 1, w.F, w.act, w.dtype)
    stack = lambda i: dev(np.stack([weights[e][i] for e in range(N)]))
    wg, wd = stack(0), stack(2)
    wu = stack(1) if w.act == "swiglu" else None
    y = new((max(A, 1), w.d), w.dtype, fill=0)
    ws = B.workspace(B.grouped_ffn_workspace_size(s))
    B.grouped_ffn(s, dev(x_perm) if A else y, dev(offsets), wg, wu, wd, y, ws)
    assert B.get_error() == B.MOE_OK
    return host_f64(y[:A])


def oracle_ffn(w, x_perm, weights, offsets):
    ref = np.zeros((w.T, w.d))
    for e in range(w.N):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            ref[a:b] = oracle.expert_rows(x_perm[a:b], *weights[e], w.act)
    return ref


def check(counts, d, F, act, dtype, seed=0):
    w, xp, ws, off = make_case(counts, d, F, act, dtype, seed)
    got = run_ffn(w, xp, ws, off)
    ref = oracle_ffn(w, xp, ws, off)
    for e in range(w.N):                              # every expert's rows on their own
        a, b = off[e], off[e + 1]
        if b > a:
            assert rel_err(got[a:b], ref[a:b]) <= tol(dtype), f"expert {e}"
    assert rel_err(got, ref) <= tol(dtype)
    return got, ref


RAGGED = [0, 1, 127, 128, 129, 300, 0, 5]
# token-tile edges: multiples of 16 and one past, 256 and one past, several tiles
RAGGED_TOKENS = [16, 17, 256, 257, 0, 31, 513, 1500]


@pytest.fixture(params=["rows", "tokens", "pairs", "rowpairs"])
def tiling(request):
    B.set_ffn_tiling(request.param)
    yield request.param
    B.set_ffn_tiling("auto")


@pytest.mark.parametrize("d,F,act", [
    (256, 384, "swiglu"),       # up: 256-wide tiles (128 gate | 128 up), down: 256-wide
    (384, 192, "swiglu"),       # up: 128-wide tiles (64 | 64), down: 128-wide
    (256, 256, "gelu_tanh"),    # up: 256-wide GELU
    (384, 384, "gelu_tanh"),    # up: 128-wide GELU, down 128-wide
    (1024, 512, "swiglu"),      # 16 K-blocks: the smem ring wraps several times
])
def test_ffn_bf16_ragged(d, F, act, tiling):
    check(RAGGED, d, F, act, "bf16", seed=d + F)
    check(RAGGED_TOKENS, d, F, act, "bf16", seed=d + F + 1)


def test_ffn_bf16_more_tiles_than_sms(tiling):
    counts = [700, 513, 64, 1, 900, 0, 333, 1500]      # 35 m-tiles x 8 n-tiles > 148
    check(counts, 512, 1024, "swiglu", "bf16", seed=3)


def test_ffn_bf16_single_expert_all_rows(tiling):
    check([0, 0, 1000, 0], 256, 256, "gelu_tanh", "bf16", seed=4)


@pytest.mark.parametrize("d,F,act", [(128, 256, "swiglu"), (36, 50, "swiglu"), (64, 100, "gelu_tanh")])
def test_ffn_f32(d, F, act):
    check([3, 0, 64, 65, 1, 130], d, F, act, "f32", seed=d)


def test_ffn_empty(tiling):
    w, xp, ws, off = make_case([0, 0, 0], 128, 64, "swiglu", "bf16", 0)
    assert run_ffn(w, xp, ws, off).shape == (0, 128)


def test_ffn_repeatable_bitwise(tiling):
    w, xp, ws, off = make_case(RAGGED, 256, 384, "swiglu", "bf16", 9)
    a = run_ffn(w, xp, ws, off)
    b = run_ffn(w, xp, ws, off)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ffn_corrupt_offsets_recorded(dtype, tiling):
    w, xp, ws, off = make_case([10, 20, 30], 128, 128, "swiglu", dtype, 0)
    bad = off.copy()
    bad[3] = 61                                       # runs past the A = 60 rows
    s = B.shape(w.T, w.d, w.N, 1, w.F, w.act, w.dtype)
    stack = lambda i: dev(np.stack([ws[e][i] for e in range(w.N)]))
    y = new((w.T, w.d), dtype, fill=0)
    wsb = B.workspace(B.grouped_ffn_workspace_size(s))
    B.grouped_ffn(s, dev(xp), dev(bad), stack(0), stack(1), stack(2), y, wsb)
    assert B.get_error() == B.MOE_ERR_CORRUPT
    assert float(y.float().abs().max()) == 0.0       # nothing written


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ffn_non_monotone_offsets_recorded(dtype):
    w, xp, ws, off = make_case([10, 20, 30], 128, 128, "swiglu", dtype, 0)
    bad = np.array([0, 20, 10, 60], dtype=np.int32)
    s = B.shape(w.T, w.d, w.N, 1, w.F, w.act, w.dtype)
    stack = lambda i: dev(np.stack([ws[e][i] for e in range(w.N)]))
    y = new((w.T, w.d), dtype, fill=0)
    B.grouped_ffn(s, dev(xp), dev(bad), stack(0), stack(1), stack(2), y,
                  B.workspace(B.grouped_ffn_workspace_size(s)))
    assert B.get_error() == B.MOE_ERR_CORRUPT
    assert float(y.float().abs().max()) == 0.0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ffn_offsets_cover_a_prefix_of_the_rows(dtype, tiling):
    """After a capacity drop the kept rows are a prefix [0, offsets[N]) of the
    A-row buffers: those rows match the oracle and the tail is not written."""
    counts = [40, 0, 129, 17]
    w, xp, ws, off = make_case(counts, 256, 256, "swiglu", dtype, 5)
    N = len(counts)
    A = w.T
    kept = off
    extra = 50                                        # rows past offsets[N], never read or written
    s = B.shape(A + extra, w.d, N, 1, w.F, w.act, w.dtype)
    stack = lambda i: dev(np.stack([ws[e][i] for e in range(N)]))
    x_full = np.concatenate([xp, xp[:extra]])
    y = new((A + extra, w.d), dtype, fill=0)
    y[A:] = 7
    B.grouped_ffn(s, dev(x_full), dev(kept), stack(0), stack(1), stack(2), y,
                  B.workspace(B.grouped_ffn_workspace_size(s)))
    assert B.get_error() == B.MOE_OK
    got = host_f64(y)
    ref = np.zeros((A, w.d))
    for e in range(N):
        a, b = kept[e], kept[e + 1]
        if b > a:
            ref[a:b] = oracle.expert_rows(xp[a:b], *ws[e], w.act)
    assert rel_err(got[:A], ref) <= tol(dtype)
    assert np.all(got[A:] == 7)


def test_tilings_agree_within_tolerance():
    """Both tensor-core tilings compute the same product (only the blocking and
    the bf16 rounding of h differ): each is within tolerance of the oracle and
    of each other."""
    w, xp, ws, off = make_case([200, 0, 300, 45, 1000], 512, 384, "swiglu", "bf16", 12)
    outs = {}
    for mode in ("rows", "tokens", "pairs", "rowpairs"):
        B.set_ffn_tiling(mode)
        outs[mode] = run_ffn(w, xp, ws, off)
    B.set_ffn_tiling("auto")
    ref = oracle_ffn(w, xp, ws, off)
    for mode, got in outs.items():
        assert rel_err(got, ref) <= tol("bf16"), mode
    assert rel_err(outs["rows"], outs["tokens"]) <= tol("bf16")
    assert rel_err(outs["pairs"], outs["tokens"]) <= tol("bf16")
    assert rel_err(outs["rowpairs"], outs["rows"]) <= tol("bf16")


@pytest.mark.parametrize("T,N,k,d,F,act", [(300, 8, 2, 256, 384, "swiglu"), (1000, 16, 4, 512, 256, "gelu_tanh"),
                                           (37, 64, 8, 256, 192, "swiglu"), (2000, 4, 2, 4096, 512, "gelu_tanh")])
def test_gathered_rows_equal_the_permuted_copy(T, N, k, d, F, act, tiling):
    """moe_grouped_ffn_gather (token rows loaded through perm by the GEMM's TMA
    gathers) gives the same bits as moe_grouped_ffn on the x_perm copy, and
    moe_permute without x_perm gives the same indices."""
    g = torch.Generator().manual_seed(T + N)
    idx = torch.stack([torch.randperm(N, generator=g)[:k] for _ in range(T)]).to(torch.int32).cuda()
    w = S.Workload("gather", T=T, d=d, N=N, k=k, F=F, act=act, dtype="bf16", seed=T)
    x = dev(S.x_all(w))
    ex = [S.expert_weights(w, e) for e in range(N)]
    WG, WD = dev(np.stack([e[0] for e in ex])), dev(np.stack([e[2] for e in ex]))
    WU = dev(np.stack([e[1] for e in ex])) if act == "swiglu" else None
    s = B.shape(T, d, N, k, F, act, "bf16")
    A = T * k
    bufs = lambda: (new((N,), "i32"), new((N + 1,), "i32"), new((A,), "i32"), new((A,), "i32"))
    ref_idx, got_idx = bufs(), bufs()
    xp = new((A, d), "bf16")
    ws = B.workspace(max(B.permute_workspace_size(s), B.grouped_ffn_workspace_size(s)))
    B.permute(s, idx, x, *ref_idx, xp, ws)
    B.permute(s, idx, x, *got_idx, None, ws)
    for a, b in zip(ref_idx, got_idx):
        assert torch.equal(a, b)
    y_ref, y_got = new((A, d), "bf16", fill=0), new((A, d), "bf16", fill=0)
    B.grouped_ffn(s, xp, ref_idx[1], WG, WU, WD, y_ref, ws)
    B.grouped_ffn_gather(s, x, got_idx[2], got_idx[1], WG, WU, WD, y_got, ws)
    assert B.get_error() == B.MOE_OK
    assert torch.equal(y_ref, y_got)


def test_gather_rejects_fp32():
    s = B.shape(4, 128, 2, 1, 64, "swiglu", "f32")
    z = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.grouped_ffn_gather(s, z, z, z, z, z, z, z, B.workspace(1 << 20))
    assert e.value.status == B.MOE_ERR_UNSUPPORTED
