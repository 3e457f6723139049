"""Benchmark of the MoE layer forward (route -> permute -> grouped FFN -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0). A step is one forward of the whole layer over
one batch of seeded synthetic tokens with the workload's shapes, through the
library's C ABI. Under torchrun every rank runs an independent replica of the
layer on its own tokens (the tokens of a batch are independent, so the work
shards by batch with no collective); value = tokens of all ranks / max time.

Default workload: the pages' worked example (4 x 2048 tokens, d 4096, 64
experts, 4096 -> 16384 -> 4096 tanh-GELU experts, top-2, bf16, fp32 gate).
--impl reference times the CPU oracle instead, on a bounded sample of the
same workload, on the host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from typing import Optional

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as S  # noqa: E402
from mixture_experts_layer_97_b300 import accounting as acc  # noqa: E402

DEFAULT_WORKLOAD = "worked-example-n64-f16384-gelu"
L2_BYTES = 126 * 1024 * 1024
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0   # nominal HBM3e bandwidth of a B300, ~8 TB/s (context fraction only)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sus=p["bf16_tflops_sustained"], src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback")


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    cs = os.path.join(ROOT, "mixture_experts_layer_97_b300", "csrc")
    for name in sorted(os.listdir(cs)):
        with open(os.path.join(cs, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


GROUPED_GEMM_SOURCES = ("common.cuh", "schedule.cuh", "ffn_tc.cuh", "ffn_tc_swap.cuh", "ffn_tc_pair.cuh")


def grouped_gemm_source_hash() -> str:
    """Hash of the sources the grouped-GEMM kernels are compiled from."""
    h = hashlib.sha1()
    cs = os.path.join(ROOT, "mixture_experts_layer_97_b300", "csrc")
    for name in GROUPED_GEMM_SOURCES:
        with open(os.path.join(cs, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload: str):
    """DRAM bytes per moe_grouped_ffn call (both GEMM launches) from a
    committed ncu capture, valid only while the grouped-GEMM sources are
    unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_hash") != grouped_gemm_source_hash():
        return None
    return rec.get("bytes_per_call")


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons. The
    sampler is started, and its first sample awaited, before the timed region;
    summary() keeps the samples taken between mark_start() and mark_end()
    (plus the one right after, which covers the region's last interval)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []          # (monotonic time, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.monotonic() + 5.0
            while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark_start(self):
        self.t0 = time.monotonic()

    def mark_end(self):
        self.t1 = time.monotonic()
        time.sleep(0.12)         # let the sample that covers the region's end arrive

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Samples between t0 and t1 (monotonic; default: mark_start / mark_end)."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0 = t0 if t0 is not None else (self.t0 if self.t0 is not None else float("-inf"))
        t1 = t1 if t1 is not None else (self.t1 if self.t1 is not None else float("inf"))
        after = [ts for ts, _ in self.lines if ts > t1]
        t1 = min(after) if after else t1      # include the first sample after the region
        for ts, ln in self.lines:
            if ts < t0 or ts > t1:
                continue
            p = [c.strip() for c in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for nm, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ replicas
def replica_workload(w: S.Workload, rank: int) -> S.Workload:
    """Rank r runs the same layer shapes on its own seeded tokens and weights
    (tokens of a batch are independent: the work shards by batch, weak scaling)."""
    return w.scaled(seed=w.seed + 1000 * rank) if rank else w


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The job's time is the slowest rank's (max over ranks; identity at N=1)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms: float) -> float:
    """Whole-job tokens/s: the tokens of all ranks over the max-over-ranks time."""
    return world * tokens_per_rank / (ms * 1e-3)


# ------------------------------------------------------------------ oracle sample
def cpu_sample_plan(w: S.Workload, target_rows: int):
    """A bounded sample of the workload for the CPU oracle: tokens whose k
    experts all lie in a small expert subset (so only that subset's weights are
    held on the host), in token order. Routing is the oracle's own."""
    import oracle
    x = S.x_all(w)
    r = oracle.route(x, S.gate_weight(w), w.k, bias=S.gate_bias(w))
    idx = r["topk_idx"]
    for n_sub in (8, 16, 24, 32, 48, w.N):
        sub = np.arange(min(n_sub, w.N))
        ok = np.all(np.isin(idx, sub), axis=1)
        toks = np.where(ok)[0]
        if toks.size * w.k >= target_rows or n_sub >= w.N:
            toks = toks[:max(1, target_rows // w.k)]
            used = np.unique(idx[toks])
            return toks, used
    raise AssertionError


def run_oracle_sample(w: S.Workload, tokens, weights: dict):
    """One oracle forward of the sampled tokens: route, every selected
    expert's FFN on its rows, combine. Returns wall seconds."""
    import oracle
    x = S.x_all(w)[tokens]
    wg, b = S.gate_weight(w), S.gate_bias(w)
    t0 = time.perf_counter()
    r = oracle.route(x, wg, w.k, bias=b)
    idx = r["topk_idx"]
    y = np.zeros((len(tokens) * w.k, w.d))
    for e in np.unique(idx):
        q, j = np.nonzero(idx == e)
        a, bb, c = weights[int(e)]
        y[q * w.k + j] = oracle.expert_rows(x[q], a, bb, c, w.act)
    oracle.combine(y, np.arange(len(tokens) * w.k, dtype=np.int32), r["topk_w"])
    return time.perf_counter() - t0


def reference_arm(args, w):
    """--impl reference: the CPU oracle timed as it stands on a bounded sample."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step_rows = {"worked-example-n64-f16384-gelu": 32, "prefill-n8-f14336": 32,
                     "zipf-skew-n128-k8": 256, "decode-t32-n64-k8": 256}.get(w.name, 64)
    tokens, used = cpu_sample_plan(w, per_step_rows)
    weights = dict(S.iter_expert_weights(w, experts=[int(e) for e in used]))
    for _ in range(args.warmup):
        run_oracle_sample(w, tokens, weights)
    times = [run_oracle_sample(w, tokens, weights) for _ in range(args.steps)]
    sec = sum(times) / len(times)
    value = len(tokens) / sec
    sample = (f"{len(tokens)} tokens of {w.name} (route + {len(tokens) * w.k} expert rows + combine) "
              f"whose experts lie in a {len(used)}-expert subset, same sample every step")
    line = {"metric": "MoE-layer tokens/s", "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "k": w.k, "d_ff": w.F, "act": w.act,
                       "sample_tokens_per_step": int(len(tokens))},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ fp32 FMA peak
def fma_peak_tflops(torch, sms: int) -> dict:
    """Measured fp32 FMA throughput of the CUDA cores (the route kernel's
    roofline denominator): the committed microbenchmark libmoe_fma_peak.so,
    scalar fma.rn.f32 and packed fma.rn.f32x2, best of 5 launches each timed
    with CUDA events on the current stream."""
    import ctypes
    from mixture_experts_layer_97_b300 import build as build_mod
    L = ctypes.CDLL(build_mod.build_fma_peak())
    L.moe_fma_peak_flops.restype = ctypes.c_double
    L.moe_fma_peak_flops.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.moe_fma_peak_launch.restype = ctypes.c_int
    L.moe_fma_peak_launch.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_void_p]
    blocks, threads, iters = sms * 8, 256, 4096
    out = torch.empty(blocks * threads, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    res = {}
    for packed, name in ((0, "fma.rn.f32"), (1, "fma.rn.f32x2")):
        best = None
        for i in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = L.moe_fma_peak_launch(ctypes.c_void_p(out.data_ptr()), blocks, threads, iters, packed,
                                       ctypes.c_void_p(stream.cuda_stream))
            b.record(stream)
            torch.cuda.synchronize()
            if rc != 0:
                raise RuntimeError(f"fma peak launch failed ({rc})")
            if i >= 2:
                ms = a.elapsed_time(b)
                best = ms if best is None else min(best, ms)
        res[name] = L.moe_fma_peak_flops(blocks, threads, iters) / (best * 1e-3) / 1e12
    res["peak"] = max(res.values())
    res["how"] = (f"{blocks} CTAs x {threads} threads, 16 independent FMA chains per thread, "
                  f"{iters * 8} steps; best of 5 launches (CUDA events)")
    return res


# ------------------------------------------------------------------ our arm
def measure(w: S.Workload, args, torch, B, world: int, rank: int, local: int, dist, want_e2e: bool,
            want_cpu: bool, steps: int, warmup: int) -> dict:
    """Upload one workload's seeded inputs, time `steps` forwards (after
    `warmup`), optionally end to end through the host-buffer entry points and
    the CPU oracle on a bounded sample. Returns the measurements (rank 0)."""
    # cpu sample plan first (host only), so its experts can be kept while uploading
    ec = args.routing == "expert"
    do_cpu = want_cpu and not ec
    if do_cpu:
        cpu_rows = {"worked-example-n64-f16384-gelu": 384, "prefill-n8-f14336": 128,
                    "zipf-skew-n128-k8": 4096, "decode-t32-n64-k8": 256}.get(w.name, 256)
        cpu_tokens, cpu_used = cpu_sample_plan(w, cpu_rows)
        keep = set(int(e) for e in cpu_used)
    else:
        keep = set()

    td = B.TORCH_DTYPE[w.dtype]
    dev = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
                     else torch.from_numpy(a)).cuda()
    x_h = S.x_all(w)
    x = dev(x_h)
    wg = dev(S.gate_weight(w))
    b_h = S.gate_bias(w)
    bias = dev(b_h) if b_h is not None else None
    WG = torch.empty((w.N, w.F, w.d), dtype=td, device="cuda")
    WU = torch.empty((w.N, w.F, w.d), dtype=td, device="cuda") if w.act == "swiglu" else None
    WD = torch.empty((w.N, w.d, w.F), dtype=td, device="cuda")
    kept = {}
    for e, (a, b_, c) in S.iter_expert_weights(w):
        WG[e].copy_(dev(a))
        if WU is not None:
            WU[e].copy_(dev(b_))
        WD[e].copy_(dev(c))
        if e in keep:
            kept[e] = (a, b_, c)
    torch.cuda.synchronize()

    s = B.shape(w.T, w.d, w.N, w.k, w.F, w.act, w.dtype)
    C = max(1, w.T * w.k // w.N) if ec else 0
    A = w.N * C if ec else w.A
    s_rows = B.shape(A, w.d, w.N, 1, w.F, w.act, w.dtype) if ec else s     # grouped FFN over the N*C rows
    s_slots = B.shape(w.T, w.d, w.N, w.N, w.F, w.act, w.dtype) if ec else s  # N (row, weight) slots per token
    if ec:
        probs = torch.empty((w.T, w.N), dtype=torch.float32, device="cuda")
        inv_ec = torch.empty((w.T, w.N), dtype=torch.int32, device="cuda")
        w_ec = torch.empty((w.T, w.N), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
    tw = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
    counts = torch.empty(w.N, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.N + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(A, dtype=torch.int32, device="cuda")
    inv = torch.empty(A, dtype=torch.int32, device="cuda")
    xp = torch.empty((A, w.d), dtype=td, device="cuda")
    yp = torch.empty((A, w.d), dtype=td, device="cuda")
    out = torch.empty((w.T, w.d), dtype=td, device="cuda")
    dropped = torch.zeros(1, dtype=torch.int32, device="cuda")
    cf = args.capacity_factor
    ws = B.workspace(max(B.permute_workspace_size(s), B.grouped_ffn_workspace_size(s_rows)))
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    flush_clean = torch.zeros(2 * L2_BYTES, dtype=torch.uint8, device="cuda")

    def flush_l2():
        """Write 2 x L2 of bytes, then read 2 x L2 of other bytes: the timed
        step starts with a cold L2 that holds no data of the layer and no
        dirty lines still to be written back."""
        flush.zero_()
        flush_clean.max()
    stream = torch.cuda.current_stream()

    def stage_route():
        if ec:
            B.route_expert_choice(s, C, x, wg, bias, probs, perm, counts, offsets, inv_ec, w_ec)
        else:
            B.route(s, x, wg, bias, idx, tw)

    # token choice: the grouping writes the permuted copy x_perm and the grouped GEMM reads it (the
    # path moe_forward takes); --gather: indices only, the first GEMM gathers the rows of x through perm
    gather = not ec and w.dtype == "bf16" and args.gather
    xp_arg = None if gather else xp

    def stage_permute():
        if ec:
            B.gather_rows(s, inv_ec, w.N, A, x, xp)
        elif cf is None:
            B.permute(s, idx, x, counts, offsets, perm, inv, xp_arg, ws)
        else:
            B.permute_capacity(s, idx, x, cf, counts, offsets, perm, inv, xp_arg, ws, dropped=dropped)

    def stage_ffn():
        if gather:
            B.grouped_ffn_gather(s_rows, x, perm, offsets, WG, WU, WD, yp, ws)
        else:
            B.grouped_ffn(s_rows, xp, offsets, WG, WU, WD, yp, ws)

    def stage_combine():
        if ec:
            B.combine(s_slots, yp, inv_ec, w_ec, out)
        else:
            B.combine(s, yp, inv, tw, out)

    stages = [stage_route, stage_permute, stage_ffn, stage_combine]

    def step(ev=None):
        for j, fn in enumerate(stages):
            if ev: ev[j].record(stream)
            fn()
        if ev: ev[4].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st = B.get_error()
    if st != B.MOE_OK:
        raise RuntimeError(f"device error during warm-up: {B.status_string(st)}")

    # Each stage captured once as a CUDA graph (the library only queues work on the caller's stream)
    # and replayed between event pairs: a stage's own launches (four for the grouping) run without
    # host gaps, and the events still give the per-stage breakdown.
    # The whole step captured once as a CUDA graph (the library only queues work on the caller's
    # stream) and replayed between two events: the step's timing. Each stage also captured on its
    # own and replayed between event pairs in separate steps: the per-stage breakdown.
    graphs = whole = None
    try:
        graphs = []
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        for fn in stages:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    fn()
            graphs.append(g)
        whole = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(whole, stream=cap):
                for fn in stages:
                    fn()
        torch.cuda.synchronize()
        for g in graphs:
            g.replay()
        whole.replay()
        torch.cuda.synchronize()
        stages = [g.replay for g in graphs]
    except RuntimeError:
        graphs = whole = None

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        clk.mark_start()
        # the timed steps: whole-step graph replays, back to back
        for i in range(steps):
            flush_l2()                         # L2 flush between timed steps (outside the events)
            wev[i][0].record(stream)
            if whole is not None:
                whole.replay()
            else:
                step()
            wev[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark_end()
        # the per-stage breakdown: as many staged steps, after a pause that lets the power state of
        # the timed steps settle (under a sustained load the part lowers its clocks at the power cap);
        # each staged step runs alone (synchronised, then a short idle gap), so its kernels are timed
        # in isolation, the condition of the burst peaks they are compared with
        time.sleep(0.5)
        ts0 = time.monotonic()
        for i in range(steps):
            flush_l2()
            step(evs[i])
            torch.cuda.synchronize()
            time.sleep(0.02)
        ts1 = time.monotonic()
        time.sleep(0.12)
        clocks_staged = clk.summary(ts0, ts1)
    if dist:
        dist.barrier()
    st = B.get_error()
    if st != B.MOE_OK:
        raise RuntimeError(f"device error during timing: {B.status_string(st)}")
    stage = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in evs])   # ms
    per_step = np.array([a.elapsed_time(b) for a, b in wev])
    staged_ms = float(np.median([e[0].elapsed_time(e[4]) for e in evs]))
    ffn_ms = float(np.median(stage[:, 2]))
    step_ms = max_over_ranks(float(np.median(per_step)), dist, "cuda")

    # end to end through the public host-buffer entry point
    e2e = None
    if want_e2e:
        x_host = torch.from_numpy(x_h.view(np.int16)).view(torch.bfloat16).pin_memory() if w.dtype == "bf16" \
            else torch.from_numpy(x_h).pin_memory()
        out_host = torch.empty((w.T, w.d), dtype=td).pin_memory()
        wsh = B.workspace(B.expert_choice_workspace_size(s, C) if ec else B.hostio_workspace_size(s))
        del ws

        def forward_e2e():
            if ec:                             # no host-buffer entry for these: copies around the call
                x.copy_(x_host, non_blocking=True)
                B.forward_expert_choice(s, C, x, wg, bias, WG, WU, WD, out, wsh)
                out_host.copy_(out, non_blocking=True)
            elif cf is None:
                B.forward_hostio(s, x_host, wg, bias, WG, WU, WD, out_host, wsh)
            else:
                x.copy_(x_host, non_blocking=True)
                B.forward_capacity(s, cf, x, wg, bias, WG, WU, WD, out, wsh)
                out_host.copy_(out, non_blocking=True)

        for _ in range(2):
            forward_e2e()
        torch.cuda.synchronize()
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps)]
        if dist:
            dist.barrier()
        for i in range(steps):
            flush_l2()
            e_ev[i][0].record(stream)
            forward_e2e()
            e_ev[i][1].record(stream)
        torch.cuda.synchronize()
        if B.get_error() != B.MOE_OK:
            raise RuntimeError("device error during the end-to-end run")
        e_ms = float(np.mean([a.elapsed_time(b) for a, b in e_ev]))
        e_ms = max_over_ranks(e_ms, dist, "cuda")
        io = w.T * w.d * w.esize
        e2e = {"value": job_throughput(w.T, world, e_ms), "unit": "tokens/s", "h2d_bytes_per_step": io,
               "d2h_bytes_per_step": io, "ms_per_step": e_ms,
               "mode": "serial: each step copies x in, runs the layer, copies out (moe_forward_hostio)"}
        if not ec and cf is None:
            # the same steps through moe_forward_hostio_pipelined: step i+1's input copy and step i-1's
            # output copy run on their own streams while step i's layer runs
            del wsh
            wsp = B.workspace(B.hostio_pipelined_workspace_size(s))
            outs_h = [out_host, torch.empty((w.T, w.d), dtype=td).pin_memory()]
            s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

            def piped(i):
                B.forward_hostio_pipelined(s, x_host, wg, bias, WG, WU, WD, outs_h[i % 2], wsp, i % 2, stream,
                                           s_in, s_out)

            for i in range(2):
                piped(i)
            torch.cuda.synchronize()
            if dist:
                dist.barrier()
            flush_l2()
            torch.cuda.synchronize()
            p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            p0.record(stream)
            s_in.wait_event(p0)
            for i in range(steps):
                piped(i)
            p1.record(s_out)                   # after the last output copy
            torch.cuda.synchronize()
            if B.get_error() != B.MOE_OK:
                raise RuntimeError("device error during the pipelined end-to-end run")
            p_ms = max_over_ranks(p0.elapsed_time(p1) / steps, dist, "cuda")
            if p_ms < e_ms:
                e2e.update({"value": job_throughput(w.T, world, p_ms), "ms_per_step": p_ms,
                            "mode": ("pipelined: moe_forward_hostio_pipelined over consecutive steps; every "
                                     "step copies its x in and its output out, overlapping the neighbouring "
                                     "steps' layer"),
                            "l2": "no flush between pipelined steps: the expert weights every step reads exceed L2"})
            e2e.update({"serial_value": job_throughput(w.T, world, e_ms), "serial_ms_per_step": e_ms,
                        "pipelined_value": job_throughput(w.T, world, p_ms), "pipelined_ms_per_step": p_ms})

    if rank != 0:
        return {}

    P = peaks()
    cnt = counts.cpu().numpy()
    # routing health of the batch, from the library's own statistics (moe_route_ex), outside the timing
    routing_stats = None
    if not ec:
        try:
            st_buf = torch.empty(B.load_stats_len(w.N), dtype=torch.float32, device="cuda")
            idx2 = torch.empty((w.T, w.k), dtype=torch.int32, device="cuda")
            tw2 = torch.empty((w.T, w.k), dtype=torch.float32, device="cuda")
            B.route_ex(s, x, wg, bias, idx2, tw2, load_stats=st_buf, ws=B.workspace(B.route_ex_workspace_size(s)))
            if B.get_error() == B.MOE_OK:
                u = B.unpack_load_stats(st_buf, w.N)
                routing_stats = {"balance_N_sum_fP": u["balance"], "activation_entropy_bits": u["entropy_bits"],
                                 "entropy_max_bits": float(np.log2(w.N)), "mean_top1_probability": u["top1"],
                                 "expert_rows": {"min": int(cnt.min()), "median": float(np.median(cnt)),
                                                 "max": int(cnt.max()), "empty": int((cnt == 0).sum())}}
        except Exception:                      # a report extra: never let it stop the benchmark line
            routing_stats = None
    rows = int(cnt.sum())                      # rows the grouped FFN computed (A unless a capacity dropped some)
    up_f, down_f = acc.up_flops(rows, w.d, w.F, w.act), acc.down_flops(rows, w.d, w.F)
    ffn_flops = up_f + down_f
    wbytes = acc.active_expert_weight_bytes(cnt, w.d, w.F, w.act, w.esize)
    # prefill-shaped (many rows per active expert): tensor roofline; decode-shaped: the HBM bytes of the
    # active experts' weights. Both fractions are reported.
    rows_per_active = rows / max(1, int((cnt > 0).sum()))
    tensor_bound = rows_per_active >= 128
    # the record is for the plain token-choice call; other routings move other bytes
    traffic = recorded_traffic(w.name) if (not ec and cf is None) else None
    tflops = ffn_flops / (ffn_ms * 1e-3) / 1e12
    gbs = wbytes / (ffn_ms * 1e-3) / 1e9
    if tensor_bound:
        roof = {"bound": "tensor", "kernel": "grouped_gemm_tc (up + down launches of moe_grouped_ffn)",
                "achieved": tflops, "peak": P["bf16"], "unit": "TFLOP/s", "frac": tflops / P["bf16"],
                "peak_kind": f"bf16 burst, {P['src']}", "frac_of_sustained": tflops / P["bf16_sus"],
                "frac_hbm_weights": gbs / P["hbm"], "traffic": traffic, "algorithmic_flops_per_call": ffn_flops,
                "algorithmic_weight_bytes_per_call": wbytes}
    else:
        roof = {"bound": "hbm", "kernel": "grouped_gemm_tc (up + down launches of moe_grouped_ffn)",
                "achieved": gbs, "peak": P["hbm"], "unit": "GB/s", "frac": gbs / P["hbm"],
                "peak_kind": f"copy bandwidth, {P['src']}", "frac_tensor": tflops / P["bf16"], "traffic": traffic,
                "algorithmic_bytes_per_call": wbytes}
    fwd_bytes = acc.decode_forward_bytes(cnt, w.T, w.d, w.N, w.k, w.F, w.act, w.esize)
    roof["forward_frac_hbm"] = fwd_bytes / (step_ms * 1e-3) / 1e9 / P["hbm"]
    # context only: against the nominal 2.25 PFLOP/s bf16 dense and ~8 TB/s HBM3e of the part
    roof["frac_of_nominal"] = (tflops / NOMINAL_BF16_TFLOPS) if tensor_bound else (gbs / NOMINAL_HBM_GBS)

    cpu = None
    if do_cpu:
        import oracle
        secs = run_oracle_sample(w, cpu_tokens, kept)
        cpu = {"value": len(cpu_tokens) / secs, "unit": "tokens/s", "cores": oracle.num_threads(),
               "kind": "oracle",
               "sample": (f"{len(cpu_tokens)} tokens (route + {len(cpu_tokens) * w.k} expert rows + combine) "
                          f"whose experts lie in a {len(cpu_used)}-expert subset; {secs:.1f} s")}
    stage_ms = {"route": float(np.median(stage[:, 0])), "permute": float(np.median(stage[:, 1])),
                "grouped_ffn": ffn_ms, "combine": float(np.median(stage[:, 3]))}
    stage_ms["staged_sum_of_stages"] = staged_ms
    return dict(w=w, C=C, ec=ec, cf=cf, gather=gather, step_ms=step_ms, ffn_ms=ffn_ms, stage_ms=stage_ms, cnt=cnt,
                ffn_flops=ffn_flops, roof=roof, cpu=cpu, e2e=e2e, clocks=clk.summary(),
                clocks_staged=clocks_staged,
                routing_stats=routing_stats, dropped=int(dropped.item()) if cf is not None else 0,
                graphs=graphs is not None, fwd_bytes=fwd_bytes, P=P)


def route_roofline(r: dict, fma: Optional[dict]) -> dict:
    """The gate projection (2 T d N fp32 FLOPs) of the route stage against the
    measured fp32 FMA peak of the CUDA cores."""
    w = r["w"]
    flops = acc.gate_flops(w.T, w.d, w.N)
    ach = flops / (r["stage_ms"]["route"] * 1e-3) / 1e12
    out = {"bound": "alu", "kernel": "route_kernel (gate GEMV/GEMM in fp32 FMA chains + top-k)", "achieved": ach,
           "unit": "TFLOP/s", "algorithmic_flops_per_call": flops, "us": r["stage_ms"]["route"] * 1e3}
    if fma:
        out.update({"peak": fma["peak"], "frac": ach / fma["peak"],
                    "peak_kind": "measured fp32 FMA (libmoe_fma_peak.so: " + fma["how"] + ")"})
    return out


def measure_ep_local(w: S.Workload, cnt: np.ndarray, torch, B, G: int, hbm_gbs: float, steps: int = 20) -> dict:
    """The receiving rank's local steps of expert parallelism (moe_ep_regroup,
    moe_ep_ungroup) at the workload's size, as if its experts were split over G
    ranks: the count table is the workload's own per-expert counts read as G
    sources x E = N / G local experts, so the rank receives all T*k rows. Each
    kernel reads and writes rows x d once (algorithmic bytes 2 rows d es); the
    all-to-all between ranks is not part of it (one GPU)."""
    E = w.N // G
    table = np.ascontiguousarray(cnt.reshape(G, E), dtype=np.int32)
    rows = int(table.sum())
    td = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    es = 2 if w.dtype == "bf16" else 4
    rc = torch.from_numpy(table.reshape(-1)).cuda()
    recv_x = torch.randn(rows, w.d, device="cuda").to(td)
    x_local = torch.empty_like(recv_x)
    y_recv = torch.empty_like(recv_x)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    src = torch.empty(rows, dtype=torch.int32, device="cuda")
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    t_re, t_un = [], []
    for i in range(steps + 3):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.zero_()
        ev[0].record(stream)
        B.ep_regroup(G, E, rc, recv_x, x_local, off, src, w.dtype)
        ev[1].record(stream)
        flush.zero_()
        ev[2].record(stream)
        B.ep_ungroup(src, x_local, y_recv, w.dtype)
        ev[3].record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            t_re.append(ev[0].elapsed_time(ev[1]))
            t_un.append(ev[2].elapsed_time(ev[3]))
    st = B.get_error()
    if st != B.MOE_OK:
        raise RuntimeError(f"device error in the expert-parallel kernels: {B.status_string(st)}")
    ok = bool(torch.equal(y_recv, recv_x))          # ungroup inverts regroup
    byt = 2 * rows * w.d * es
    re_ms, un_ms = float(np.median(t_re)), float(np.median(t_un))
    return {"ranks": G, "local_experts": E, "rows": rows, "algorithmic_bytes_per_kernel": byt,
            "regroup_us": re_ms * 1e3, "ungroup_us": un_ms * 1e3,
            "regroup_gbs": byt / (re_ms * 1e-3) / 1e9, "ungroup_gbs": byt / (un_ms * 1e-3) / 1e9,
            "regroup_frac_hbm": byt / (re_ms * 1e-3) / 1e9 / hbm_gbs,
            "ungroup_frac_hbm": byt / (un_ms * 1e-3) / 1e9 / hbm_gbs,
            "peak_gbs": hbm_gbs, "ungroup_inverts_regroup": ok,
            "timing": f"median of {steps} launches each, CUDA events, L2 flushed before each launch"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(S.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gather", action="store_true",
                    help="grouping without x_perm; the grouped GEMM gathers token rows through perm")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-shaped sub-record that follows the headline workload")
    ap.add_argument("--ffn-tiling", default="auto", choices=["auto", "rows", "tokens", "pairs", "rowpairs"],
                    help="tensor-core tiling of the grouped GEMMs (library default: auto)")
    ap.add_argument("--capacity-factor", type=float, default=None,
                    help="expert capacity ceil(cf * T * k / N); overflow assignments are dropped")
    ap.add_argument("--routing", default="token", choices=["token", "expert"],
                    help="token choice (top-k per token) or expert choice (each expert takes C = T*k/N tokens)")
    args = ap.parse_args()
    if args.routing == "expert" and args.capacity_factor is not None:
        ap.error("--capacity-factor applies to token-choice routing only")
    args.warmup = max(args.warmup, 3)
    w0 = S.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w0)

    import torch
    from mixture_experts_layer_97_b300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    B.set_ffn_tiling(args.ffn_tiling)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    w = replica_workload(w0, rank)
    r = measure(w, args, torch, B, world, rank, local, dist, want_e2e=not args.no_e2e,
                want_cpu=rank == 0 and not args.no_cpu_baseline, steps=args.steps, warmup=args.warmup)
    fma = None
    if rank == 0:
        try:
            fma = fma_peak_tflops(torch, torch.cuda.get_device_properties(local).multi_processor_count)
        except (OSError, RuntimeError):
            fma = None
    # the expert-parallel receiving rank's local kernels at the headline workload's size (8 ranks)
    ep_local = None
    if rank == 0 and w.N % 8 == 0 and args.routing == "token" and args.capacity_factor is None:
        try:
            ep_local = measure_ep_local(w, r["cnt"], torch, B, 8, r["P"]["hbm"])
        except (RuntimeError, torch.cuda.OutOfMemoryError) as exc:   # a side record: never costs the line
            ep_local = {"error": str(exc).splitlines()[0]}
    # the decode-shaped layer (HBM-bound on its active experts' weights), timed after the headline run
    dec = None
    decode_name = "decode-t32-n64-k8"
    if not args.no_decode and w0.name != decode_name and args.routing == "token" and args.capacity_factor is None:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        wd = replica_workload(S.WORKLOADS[decode_name], rank)
        rd = measure(wd, args, torch, B, world, rank, local, dist, want_e2e=not args.no_e2e,
                     want_cpu=rank == 0 and not args.no_cpu_baseline, steps=max(args.steps, 50),
                     warmup=max(args.warmup, 10))
        if rank == 0:
            dec = {"workload": decode_name, "ms_per_step": rd["step_ms"],
                   "value": job_throughput(wd.T, world, rd["step_ms"]), "unit": "tokens/s",
                   "stage_ms": rd["stage_ms"],
                   "ffn_gbs": rd["roof"]["achieved"] if rd["roof"]["bound"] == "hbm" else None,
                   "ffn_frac_hbm": rd["roof"]["frac"] if rd["roof"]["bound"] == "hbm" else None,
                   "forward_frac_hbm": rd["roof"]["forward_frac_hbm"],
                   "forward_algorithmic_bytes": rd["fwd_bytes"], "peak_gbs": rd["P"]["hbm"],
                   "active_experts": int((rd["cnt"] > 0).sum()), "route_roofline": route_roofline(rd, fma),
                   "clocks": rd["clocks"], "clocks_staged": rd["clocks_staged"], "cpu_baseline": rd["cpu"],
                   "e2e": rd["e2e"],
                   "steps": max(args.steps, 50), "warmup": max(args.warmup, 10)}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    C, ec, cf = r["C"], r["ec"], r["cf"]
    cnt = r["cnt"]
    line = {
        "metric": "MoE-layer tokens/s", "value": job_throughput(w.T, world, r["step_ms"]), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "N": w.N, "k": w.k, "d_ff": w.F, "act": w.act,
                   "gate": "fp32", "ffn_tiling": args.ffn_tiling, "capacity_factor": cf,
                   "token_rows": "gathered by the grouped GEMM through perm" if r["gather"] else "x_perm copy",
                   "routing": "expert choice, C = T*k/N = %d tokens per expert" % C if ec else "token choice (top-k)", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (2 x 126 MB write, then 2 x 126 MB read of another buffer); expert weights also exceed L2"},
        "timing": ("median over the timed steps, each one CUDA-graph replay of the whole step between two CUDA "
                   "events on the stream; stage_ms: median over as many later steps (after a 0.5 s pause), each "
                   "run alone (synchronised, 20 ms apart), in which each stage is its own graph replay between "
                   "event pairs (their sum, staged_sum_of_stages, adds the gaps between replays); the roofline "
                   "fractions use these stage times, clocks_staged their clock record"
                   if r["graphs"] else "median over steps of eager stage calls between CUDA events"),
        "ffn_tflops": r["ffn_flops"] / (r["ffn_ms"] * 1e-3) / 1e12,
        "layer_tflops": acc.layer_flops(w.T, w.d, w.N, w.k, w.F, w.act) / (r["step_ms"] * 1e-3) / 1e12,
        "stage_ms": r["stage_ms"],
        "active_experts": int((cnt > 0).sum()), "max_expert_rows": int(cnt.max()),
        "routing_stats": r["routing_stats"], "dropped_assignments": r["dropped"],
        "roofline": r["roof"], "route_roofline": route_roofline(r, fma), "fma_peak": fma,
        "cpu_baseline": r["cpu"], "e2e": r["e2e"],
        # per step: token choice: route 1 + grouping (1 launch for T*k <= 2048, else hist, scan, rank and the
        # row copy unless gathered) + grouped FFN 2 + combine 1; expert choice: route 1 + select 1 + row copy 1
        # + grouped FFN 2 + combine 1 (the tile-counter memsets of the SM-pair GEMM are not kernels)
        "gpu_launches": args.steps * (6 if ec else (1 + (1 if w.T * w.k <= 2048 else (3 if r["gather"] else 4))
                                                        + 2 + 1)),
        "clocks": r["clocks"],
        "clocks_staged": r["clocks_staged"],
        "ep_local": ep_local,
        "decode": dec,
        "kernel_source": kernel_source_hash(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
