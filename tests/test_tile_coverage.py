"""Host checks of the stratified row sets used by the full-size parity tests:
for any per-expert row counts, the set hits every block of both grouped-GEMM
tilings (row tiles; token tiles and their SM-pair halves), and the host
restatement of the token-tile rule partitions each expert's rows."""
import numpy as np
import pytest

from tests import tiles

EDGE = [0, 1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 213, 255, 256, 257, 300, 319, 511, 512, 513, 767, 768,
        769, 1024, 1025, 4097, 16245]


@pytest.mark.parametrize("c", EDGE)
def test_token_tiles_partition_the_rows(c):
    t = tiles.token_tiles(c)
    covered = []
    for lo, hi, nt in t:
        assert 0 < hi - lo <= tiles.TOKEN_TILE_MAX
        assert nt % 16 == 0 and nt >= hi - lo and nt - (hi - lo) < 16
        covered.extend(range(lo, hi))
    assert covered == list(range(c))
    if c:
        assert len(t) == -(-c // 256)


@pytest.mark.parametrize("seed", range(6))
def test_stratified_rows_cover_every_block(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 200))
    counts = np.concatenate([rng.choice(EDGE, size=N // 2), rng.integers(0, 3000, size=N - N // 2)])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows = tiles.stratified_rows(offsets)
    assert np.all(np.diff(rows) > 0)
    assert tiles.uncovered(counts, offsets, rows) == []
    # the set stays a small fraction of the rows for large experts
    big = counts >= 1024
    if big.any():
        assert len(rows) < 0.1 * offsets[-1] + 20 * N


def test_a_set_missing_a_block_is_detected():
    counts = np.array([300, 0, 20])
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows = tiles.stratified_rows(offsets)
    # drop every row of expert 0's second token tile (rows 160..299)
    keep = rows[(rows < 160) | (rows >= 300)]
    miss = tiles.uncovered(counts, offsets, keep)
    assert any(kind == "token" and lo == 160 for _, kind, lo, _ in miss)
