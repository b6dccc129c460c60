"""Pins of the oracle's load-balancing split (Grendel-GS notes §3.1) and scheduling order
(Odin summary: relative locality graph, Jaccard weights, s(v | U_prev) = sum of w_uv), CPU only.

Each check comes from something other than the oracle's own loops: numpy's block sums,
cumsum and searchsorted (exact here: the totals are far below 2^52), closed forms of uniform
and degenerate profiles, a balance bound any split at the K-quantiles must meet, and orders
worked by hand on block-structured weights.
"""
import numpy as np
import pytest

import oracle


def _blocks(cost):
    """Per-tile sums of a H x W map with numpy: zero-pad to a multiple of 16, reshape, sum."""
    H, W = cost.shape
    Ty, Tx = (H + 15) // 16, (W + 15) // 16
    pad = np.zeros((Ty * 16, Tx * 16), np.uint64)
    pad[:H, :W] = cost
    return pad.reshape(Ty, 16, Tx, 16).sum(axis=(1, 3)).ravel()


@pytest.mark.parametrize("H,W,K,seed", [(40, 50, 4, 0), (128, 128, 3, 1), (820, 1236, 8, 2), (17, 33, 5, 3)])
def test_tile_split_matches_numpy(H, W, K, seed):
    rng = np.random.default_rng(seed)
    cost = rng.integers(0, 10_000, size=(H, W), dtype=np.uint32)
    cost[rng.random((H, W)) < 0.3] = 0  # empty regions (sky)
    tc, cum, bounds = oracle.tile_split(cost, K)
    assert np.array_equal(tc, _blocks(cost))
    assert np.array_equal(cum, np.cumsum(_blocks(cost)))
    total = float(cum[-1])
    want = [0] + [int(np.searchsorted(cum.astype(np.float64), k * total / K, side="right")) for k in range(1, K)]
    assert np.array_equal(bounds, np.array(want + [len(tc)]))
    # balance: every part holds at most Total / K plus one tile's cost
    part = [int(tc[bounds[k]:bounds[k + 1]].sum()) for k in range(K)]
    assert sum(part) == int(cum[-1])
    assert max(part) <= total / K + int(tc.max())


def test_tile_split_closed_forms():
    # uniform cost, T divisible by K: equal parts
    c = np.full((64, 96), 3, np.uint32)  # 4 x 6 = 24 tiles of 768
    _, _, b = oracle.tile_split(c, 4)
    assert b.tolist() == [0, 6, 12, 18, 24]
    # one part: everything
    _, _, b = oracle.tile_split(c, 1)
    assert b.tolist() == [0, 24]
    # no cost at all: every tile's cumulative cost is at most every target, so the first part
    # takes every tile
    _, cum, b = oracle.tile_split(np.zeros((32, 32), np.uint32), 3)
    assert not cum.any() and b.tolist() == [0, 4, 4, 4]
    # all the cost in the last tile: the first K - 1 splits sit before it
    c = np.zeros((32, 48), np.uint32)
    c[20, 40] = 100
    _, _, b = oracle.tile_split(c, 3)
    assert b.tolist() == [0, 5, 5, 6]


def test_view_order_two_clusters():
    # views {0, 1} and {2, 3} see overlapping primitives, the clusters none: the weakest
    # transition alternates between the clusters
    w = np.array([[1, .9, 0, 0], [.9, 1, 0, 0], [0, 0, 1, .8], [0, 0, .8, 1]], np.float32)
    order, score = oracle.view_order(w, unit=1)
    assert order.tolist() == [0, 2, 1, 3] and not score.any()


def test_view_order_chain():
    # views on a line, neighbours sharing half their primitives: 0, then 2 (0 shares with 1),
    # then 4 (2 shares with 1 and 3), then 1, then 3
    B = 5
    w = np.eye(B, dtype=np.float32)
    for i in range(B - 1):
        w[i, i + 1] = w[i + 1, i] = 0.5
    order, score = oracle.view_order(w, unit=1)
    assert order.tolist() == [0, 2, 4, 1, 3] and not score.any()


@pytest.mark.parametrize("unit", [1, 2, 3])
def test_view_order_equal_weights(unit):
    # every pair equally coupled: all ties, so index order; a view's score is c times the
    # size of the previous unit (0 in the first unit)
    B, c = 7, np.float32(0.25)
    w = np.full((B, B), c, np.float32)
    np.fill_diagonal(w, 1)
    order, score = oracle.view_order(w, unit=unit)
    assert order.tolist() == list(range(B))
    assert score.tolist() == [0.0 if k < unit else float(c * unit) for k in range(B)]


def test_view_order_single_view_and_unit_covering_all():
    order, score = oracle.view_order(np.ones((1, 1), np.float32), unit=1)
    assert order.tolist() == [0] and score.tolist() == [0.0]
    w = np.random.default_rng(4).random((6, 6)).astype(np.float32)
    order, _ = oracle.view_order(w, unit=6)  # one unit: no previous set, index order
    assert order.tolist() == list(range(6))


# ------------------------------------------------------------------ opacity pruning
def test_prune_matches_boolean_indexing():
    rng = np.random.default_rng(5)
    P = rng.standard_normal((15, 1000, 4)).astype(np.float32)
    M = rng.standard_normal((15, 1000, 4)).astype(np.float32)
    V = rng.random((15, 1000, 4)).astype(np.float32)
    P[0, 7, 3] = np.nan  # a NaN logit is not >= any threshold
    t = np.float32(-0.3)
    P[0, 11, 3] = t  # exactly on the threshold: kept
    k, (Po, Mo, Vo) = oracle.prune([P, M, V], float(t))
    keep = P[0, :, 3] >= t
    assert keep[11] and not keep[7]
    assert k == int(keep.sum())
    for got, src in ((Po, P), (Mo, M), (Vo, V)):
        assert np.array_equal(got, src[:, keep])


def test_prune_closed_forms():
    P = np.random.default_rng(6).standard_normal((15, 50, 4)).astype(np.float32)
    k, (Po,) = oracle.prune([P], -np.inf)
    assert k == 50 and np.array_equal(Po, P)  # nothing below -inf: identity
    k, (Po,) = oracle.prune([P], np.inf)
    assert k == 0 and Po.shape == (15, 0, 4)
    k, _ = oracle.prune([np.zeros((15, 0, 4), np.float32)], 0.0)
    assert k == 0
