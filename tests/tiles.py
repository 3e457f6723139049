"""The grouped GEMMs' tile schedule, restated on the host, and the stratified
row sets the full-size parity tests compare against the oracle.

The grouped GEMM ("MoE显存与计算开销四阶段手算指南" section 4.3: one launch over
all experts' contiguous rows with expert offsets) blocks each expert's rows in
one of two ways, and the full-size tests must compare at least one row of
every block the kernels produce:

  row tiles     an expert's c rows in 128-row tiles [128 i, min(c, 128 (i+1)));
                on SM pairs a 256-row tile's two CTAs hold its 128-row halves,
                which are exactly these 128-row blocks
  token tiles   ntt = ceil(c / 256) tiles of base = roundup16(ceil(c / ntt))
                rows, tile i = [i base, min(c, (i+1) base)); the MMA's N side
                is the tile's rows rounded up to 16 (nt). On SM pairs each CTA
                holds one half of the tile's nt rows: [0, nt/2) and
                [nt/2, nt), so both halves are blocks of their own.

Each block is a (expert, kind, lo, hi) unit of local rows; the feature
dimension needs no sampling, since every compared row is compared over all of
its columns (all d outputs; all F hidden units when h is compared).
"""
from __future__ import annotations

import numpy as np

ROW_TILE = 128
TOKEN_TILE_MAX = 256


def row_tiles(c: int):
    return [(lo, min(c, lo + ROW_TILE)) for lo in range(0, c, ROW_TILE)]


def token_tiles(c: int):
    """(lo, hi, nt) of each token tile of an expert with c rows."""
    if c <= 0:
        return []
    ntt = -(-c // TOKEN_TILE_MAX)
    base = ((-(-c // ntt)) + 15) & ~15
    out = []
    for i in range(ntt):
        lo = i * base
        hi = min(c, lo + base)
        if hi > lo:
            out.append((lo, hi, (hi - lo + 15) & ~15))
    return out


def units(counts):
    """Every block of every expert's rows under both tilings (local rows)."""
    out = []
    for e, c in enumerate(np.asarray(counts).tolist()):
        for lo, hi in row_tiles(c):
            out.append((e, "row", lo, hi))
        for lo, hi, nt in token_tiles(c):
            half = nt // 2
            out.append((e, "token", lo, hi))
            out.append((e, "pair-half0", lo, min(hi, lo + half)))
            if lo + half < hi:
                out.append((e, "pair-half1", lo + half, hi))
    return out


def stratified_local_rows(c: int):
    """Local rows of one expert that hit every block of both tilings: the
    first and last row of the expert and of every block, and rows 255, 256,
    257, 511, 512 where they exist."""
    rows = {0, c - 1}
    for lo, hi in row_tiles(c):
        rows |= {lo, hi - 1}
    for lo, hi, nt in token_tiles(c):
        rows |= {lo, hi - 1}
        m = lo + nt // 2
        if m < hi:
            rows |= {m - 1, m}
    rows |= {255, 256, 257, 511, 512}
    return sorted(r for r in rows if 0 <= r < c)


def stratified_rows(offsets):
    """Global rows (into x_perm / h / y_perm) of the stratified set."""
    off = np.asarray(offsets, dtype=np.int64)
    out = []
    for e in range(len(off) - 1):
        c = int(off[e + 1] - off[e])
        out.extend(int(off[e]) + r for r in stratified_local_rows(c))
    return np.asarray(out, dtype=np.int64)


def uncovered(counts, offsets, rows):
    """Units that hold none of the given global rows."""
    off = np.asarray(offsets, dtype=np.int64)
    have = np.zeros(int(off[-1]), dtype=bool)
    have[np.asarray(rows, dtype=np.int64)] = True
    missing = []
    for e, kind, lo, hi in units(counts):
        if not have[off[e] + lo:off[e] + hi].any():
            missing.append((e, kind, lo, hi))
    return missing
