"""Host logic of bench.py without a GPU: the replica (multi-rank) arithmetic
under a real two-process gloo group, and the clock-sample summary."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import moe_synth as S


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.replica_workload(S.WORKLOADS["decode-t32-n64-k8"], rank)
        ms = 1.0 + rank                       # rank 1 is the slow one
        t = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = (w.seed, t, bench.job_throughput(w.T, world, t))
    finally:
        dist.destroy_process_group()


def test_replicas_max_over_ranks_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                               # each rank its own tokens
    assert all(res[r][1] == 2.0 for r in range(world))       # the slowest rank's time
    assert all(res[r][2] == pytest.approx(world * 32 / 2e-3) for r in range(world))


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    w = S.WORKLOADS["tiny-f32"]
    assert bench.replica_workload(w, 0) is w
    assert bench.job_throughput(64, 1, 2.0) == pytest.approx(32000.0)


def test_clock_summary_parses_and_flags_throttling():
    c = bench.ClockSampler(0)
    c.lines = [(0.9, "0, 1000, 2032, 300.0, 0x0, Not Active, Not Active, Active, Not Active"),   # before the region
               (1.1, "0, 1900, 2032, 900.0, 0x4, Not Active, Not Active, Not Active, Active"),
               (1.2, "0, 2000, 2032, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active"),
               (1.3, "0, 1950, 2032, 980.0, 0x0, Active, Not Active, Not Active, Not Active"),
               (1.35, "garbage"),
               (1.45, "0, 1960, 2032, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active"),  # covers the end
               (1.6, "0, 500, 2032, 100.0, 0x0, Not Active, Active, Not Active, Not Active")]      # after
    c.t0, c.t1 = 1.0, 1.4
    r = c.summary()
    assert r["sm_mhz"] == 1955 and r["sm_max_mhz"] == 2032 and r["samples"] == 4
    assert r["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0
