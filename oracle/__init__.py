"""CPU oracle of the MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Everything is computed in fp64 except the gate logits, which the pages keep in
fp32 ("MoE混合专家模型计算原理与推理部署实战解析" sections 2.4 and 7): the top-k
decision is taken on the plain fp32 evaluation of x @ W_g (a sequential FMA
chain in index order), so that an fp32 kernel can be held to bit-exact
routing. gate="fp64" gives the exact-logit decision for comparison.

Only the tests, the package smoke check and the benchmark's CPU baseline may
import this package. The CUDA library never links, loads or calls it, and it
imports nothing from the CUDA package; the one module both sides use is the
seeded input generator ``moe_synth``.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64, loops), compiled with
gcc into ``liboracle_moe.so`` beside it. This wrapper only marshals numpy
arrays. Parity status of each function (what pins it) is stated in the test
suite's oracle pin tests; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_moe.so")

F64, F32, BF16 = 0, 1, 2
SWIGLU, GELU_TANH = 0, 1
ACTS = {"swiglu": SWIGLU, "gelu_tanh": GELU_TANH}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP). Returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.oracle_num_threads.restype = I
        L.oracle_route.argtypes = [I64, I, I, I, P, I, P, I, P, I, I, I, P, P, P, P, P, P]
        L.oracle_route.restype = I
        L.oracle_permute.argtypes = [I64, I, I, P, P, P, P, P]
        L.oracle_permute.restype = I
        L.oracle_capacity.argtypes = [I64, I, I, ctypes.c_double]
        L.oracle_capacity.restype = I64
        L.oracle_permute_capacity.argtypes = [I64, I, I, P, I64, P, P, P, P]
        L.oracle_permute_capacity.restype = I64
        L.oracle_expert_rows.argtypes = [I64, I, I, I, P, I, P, P, P, I, P, P]
        L.oracle_expert_rows.restype = I
        L.oracle_combine.argtypes = [I64, P, I, I, P, P, P, P]
        L.oracle_combine.restype = I
        L.oracle_expert_choice.argtypes = [I64, I, I64, P, P, P, P, P, P, P]
        L.oracle_expert_choice.restype = I
        L.oracle_load_stats.argtypes = [I64, I, I, P, P, P, P, P]
        L.oracle_load_stats.restype = I
        L.oracle_forward.argtypes = [I64, I, I, I, I, I, P, I, P, I, P, I, I, I, P, P, P, I,
                                     P, P, P, P, P, P, P, P, P]
        L.oracle_forward.restype = I
        L.oracle_ep_regroup.argtypes = [I, I, P, P, P]
        L.oracle_ep_regroup.restype = I
        _lib = L
    return _lib


def num_threads() -> int:
    return lib().oracle_num_threads()


def _dt(a: Optional[np.ndarray]) -> int:
    if a is None:
        return F64
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle input dtype {a.dtype} (want f64, f32 or bf16 bits as uint16)")


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


def _p(a):
    return None if a is None else a.ctypes.data


BIAS_MODES = {"logits": 0, "select": 1}


def route(x, wg, k, bias=None, want_logits=False, gate="fp32", bias_mode="logits", want_probs=False):
    """Gate -> softmax -> top-k -> renormalise for every row of x.

    gate="fp32" (the pages' precision for the gate) takes the top-k decision
    on the fp32 logits of the sequential FMA chain; gate="fp64" on exact
    logits. bias_mode="logits" adds the bias to the logits before the
    softmax; "select" adds it only to the scores that choose the experts.
    Returns dict(topk_idx [T,k] int32, topk_w [T,k] f64, cert [T], errb [T,N]
    (both about the exact scores), and logits [T,N] (the scores) / probs
    [T,N] (the softmax) when asked)."""
    x, wg, bias = _c(x), _c(wg), _c(bias)
    T, d = x.shape
    N = wg.shape[1]
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    cert = np.empty((T,), np.float64)
    errb = np.empty((T, N), np.float64)
    logits = np.empty((T, N), np.float64) if want_logits else None
    probs = np.empty((T, N), np.float64) if want_probs else None
    rc = lib().oracle_route(T, d, N, k, _p(x), _dt(x), _p(wg), _dt(wg), _p(bias), _dt(bias), BIAS_MODES[bias_mode],
                            1 if gate == "fp32" else 0, _p(idx), _p(w), _p(logits), _p(errb), _p(cert), _p(probs))
    if rc:
        raise ValueError("oracle_route: bad arguments")
    out = dict(topk_idx=idx, topk_w=w, cert=cert, errb=errb)
    if want_logits:
        out["logits"] = logits
    if want_probs:
        out["probs"] = probs
    return out


def load_stats(probs, topk_idx):
    """Routing statistics of one batch: f [N] (fraction of assignments per
    expert), P [N] (mean gate probability), balance = N * sum f*P, entropy
    (bits) of f, top1 = mean max probability."""
    probs = np.ascontiguousarray(probs, dtype=np.float64)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, N = probs.shape
    k = idx.shape[1] if idx.ndim == 2 else 1
    f = np.empty(N, np.float64)
    P = np.empty(N, np.float64)
    o = np.empty(3, np.float64)
    if lib().oracle_load_stats(T, N, k, _p(probs), _p(idx), _p(f), _p(P), _p(o)):
        raise ValueError("oracle_load_stats: expert index out of range")
    return dict(f=f, P=P, balance=float(o[0]), entropy_bits=float(o[1]), top1=float(o[2]))


def permute(topk_idx, N):
    """Counts, offsets, perm (row -> token) and inv_perm (t*k+j -> row)."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(N, np.int32)
    offsets = np.empty(N + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    inv = np.empty(T * k, np.int32)
    rc = lib().oracle_permute(T, N, k, _p(idx), _p(counts), _p(offsets), _p(perm), _p(inv))
    if rc:
        raise ValueError("oracle_permute: expert index out of range")
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv)


def capacity(T, N, k, capacity_factor) -> int:
    """Rows an expert may take: ceil(capacity_factor * T * k / N)."""
    return int(lib().oracle_capacity(T, N, k, float(capacity_factor)))


def permute_capacity(topk_idx, N, cap):
    """Grouping with an expert capacity: kept counts, offsets, perm and
    inv_perm (-2 for a dropped assignment), and the number dropped."""
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(N, np.int32)
    offsets = np.empty(N + 1, np.int32)
    perm = np.full(T * k, -1, np.int32)
    inv = np.empty(T * k, np.int32)
    dropped = lib().oracle_permute_capacity(T, N, k, _p(idx), int(cap), _p(counts), _p(offsets), _p(perm), _p(inv))
    if dropped < 0:
        raise ValueError("oracle_permute_capacity: expert index out of range")
    kept = int(offsets[N])
    return dict(counts=counts, offsets=offsets, perm=perm[:kept], inv_perm=inv, dropped=int(dropped))


def expert_choice(probs, C):
    """Expert-choice routing on the gate probabilities [T, N]: each expert
    takes its C most probable tokens (equal -> lower token id). Returns
    perm [N*C] (row -> token, expert e's rows e*C.. in ascending token
    order), w_row [N*C], inv [T, N] (row or -2), w [T, N] (p or 0), and per
    expert thr (smallest value picked) / next (largest value left, -1 when
    C == T)."""
    probs = np.ascontiguousarray(probs, dtype=np.float64)
    T, N = probs.shape
    C = int(C)
    perm = np.empty(max(N * C, 1), np.int32)
    w_row = np.empty(max(N * C, 1), np.float64)
    inv = np.empty((T, N), np.int32)
    w = np.empty((T, N), np.float64)
    thr = np.empty(N, np.float64)
    nxt = np.empty(N, np.float64)
    if lib().oracle_expert_choice(T, N, C, _p(probs), _p(perm), _p(w_row), _p(inv), _p(w), _p(thr), _p(nxt)):
        raise ValueError("oracle_expert_choice: bad arguments (need 0 <= C <= T)")
    return dict(perm=perm[:N * C], w_row=w_row[:N * C], inv=inv, w=w, thr=thr, next=nxt)


def ep_regroup(recv_counts):
    """Expert parallelism, receiving side: the rows received from G source
    cards, ordered (source g, local expert e, source order) with
    recv_counts[g, e] rows per run, ordered instead by (e, g, source order).
    Returns offsets_local [E+1] and local_src [rows] (the received row each
    local row takes)."""
    rc = np.ascontiguousarray(recv_counts, dtype=np.int32)
    G, E = rc.shape
    rows = int(rc.sum())
    offsets = np.empty(E + 1, np.int32)
    src = np.empty(max(rows, 1), np.int32)
    if lib().oracle_ep_regroup(G, E, _p(rc), _p(offsets), _p(src)):
        raise ValueError("oracle_ep_regroup: negative count")
    return dict(offsets_local=offsets, local_src=src[:rows])


def expert_rows(x_rows, w_gate, w_up, w_down, act, want_h=False):
    """One expert's FFN on rows [n, d]; weights [F,d], [F,d] or None, [d,F]."""
    x_rows, w_gate, w_up, w_down = _c(x_rows), _c(w_gate), _c(w_up), _c(w_down)
    n, d = x_rows.shape
    F = w_gate.shape[0]
    wdt = _dt(w_gate)
    y = np.empty((n, d), np.float64)
    h = np.empty((n, F), np.float64) if want_h else None
    rc = lib().oracle_expert_rows(n, d, F, ACTS[act], _p(x_rows), _dt(x_rows), _p(w_gate), _p(w_up),
                                  _p(w_down), wdt, _p(y), _p(h))
    if rc:
        raise ValueError("oracle_expert_rows: bad arguments")
    return (y, h) if want_h else y


def combine(y_perm, inv_perm, topk_w, tokens=None):
    """out[t] = sum_j w[t,j] * y_perm[inv_perm[t*k+j]] for the listed tokens."""
    y_perm = np.ascontiguousarray(y_perm, dtype=np.float64)
    inv = np.ascontiguousarray(inv_perm, dtype=np.int32).reshape(-1)
    w = np.ascontiguousarray(topk_w, dtype=np.float64)
    T, k = w.shape
    d = y_perm.shape[1]
    tok = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int64)
    n = T if tok is None else tok.shape[0]
    out = np.empty((n, d), np.float64)
    lib().oracle_combine(n, _p(tok), d, k, _p(y_perm), _p(inv), _p(w), _p(out))
    return out


def forward(x, wg, bias, w_gate, w_up, w_down, k, act, gate="fp32", bias_mode="logits"):
    """The whole layer: route -> permute -> per-expert FFN -> combine."""
    x, wg, bias, w_gate, w_up, w_down = map(_c, (x, wg, bias, w_gate, w_up, w_down))
    T, d = x.shape
    N = wg.shape[1]
    F = w_gate.shape[1]
    A = T * k
    r = dict(topk_idx=np.empty((T, k), np.int32), topk_w=np.empty((T, k), np.float64),
             cert=np.empty(T, np.float64), counts=np.empty(N, np.int32),
             offsets=np.empty(N + 1, np.int32), perm=np.empty(A, np.int32),
             inv_perm=np.empty(A, np.int32), y_perm=np.empty((A, d), np.float64),
             out=np.empty((T, d), np.float64))
    rc = lib().oracle_forward(T, d, N, k, F, ACTS[act], _p(x), _dt(x), _p(wg), _dt(wg), _p(bias), _dt(bias),
                              BIAS_MODES[bias_mode], 1 if gate == "fp32" else 0, _p(w_gate), _p(w_up), _p(w_down), _dt(w_gate),
                              _p(r["topk_idx"]), _p(r["topk_w"]), _p(r["cert"]), _p(r["counts"]),
                              _p(r["offsets"]), _p(r["perm"]), _p(r["inv_perm"]), _p(r["y_perm"]),
                              _p(r["out"]))
    if rc:
        raise ValueError("oracle_forward failed")
    return r
