"""Pins of the oracle's expert-parallel regrouping (oracle.ep_regroup), which
the GPU kernel is compared with bit for bit: against a stable sort of the
received rows by (local expert, source card) -- a library routine restating
the same order -- against the identity for one card, and by its invariants."""
import numpy as np
import pytest

import oracle


def _by_sort(rc):
    """Received rows tagged (g, e) in arrival order, stably sorted by (e, g)."""
    G, E = rc.shape
    tags_g = np.repeat(np.repeat(np.arange(G), E), rc.reshape(-1))
    tags_e = np.repeat(np.tile(np.arange(E), G), rc.reshape(-1))
    order = np.lexsort((tags_g, tags_e))            # primary e, then g; stable keeps source order
    counts_e = rc.sum(axis=0)
    return np.concatenate([[0], np.cumsum(counts_e)]), order


@pytest.mark.parametrize("seed", range(8))
def test_regroup_equals_stable_sort_by_expert_then_source(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.integers(1, 9))
    E = int(rng.integers(1, 9))
    rc = rng.integers(0, 6, size=(G, E)) * (rng.random((G, E)) < 0.7)
    r = oracle.ep_regroup(rc)
    off, order = _by_sort(rc)
    np.testing.assert_array_equal(r["offsets_local"], off)
    np.testing.assert_array_equal(r["local_src"], order)


def test_regroup_one_card_is_the_identity():
    rc = np.array([[3, 0, 5, 1]])
    r = oracle.ep_regroup(rc)
    np.testing.assert_array_equal(r["local_src"], np.arange(9))
    np.testing.assert_array_equal(r["offsets_local"], [0, 3, 3, 8, 9])


def test_regroup_hand_case_and_bijection():
    # received: g0 -> e0 rows 0,1; e2 row 2.  g1 -> e0 row 3; e1 rows 4,5,6
    rc = np.array([[2, 0, 1], [1, 3, 0]])
    r = oracle.ep_regroup(rc)
    np.testing.assert_array_equal(r["offsets_local"], [0, 3, 6, 7])
    np.testing.assert_array_equal(r["local_src"], [0, 1, 3, 4, 5, 6, 2])
    assert sorted(r["local_src"].tolist()) == list(range(7))


def test_regroup_empty_and_negative():
    r = oracle.ep_regroup(np.zeros((3, 2), dtype=np.int32))
    assert r["local_src"].size == 0 and r["offsets_local"].tolist() == [0, 0, 0]
    with pytest.raises(ValueError):
        oracle.ep_regroup(np.array([[1, -1]]))
