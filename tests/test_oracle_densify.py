"""Pins of the oracle's densification (clone / split) and of its statistic.

Grendel-GS notes, 训练流程 ("致密化": clone or split Gaussians that need more detail).  The
readings (the pages give no criterion): selected when the mean over the views that see a
Gaussian of its screen-space mean-gradient length reaches a threshold; split when its largest
log-scale exceeds a threshold, else cloned; split children at mu + R(q)(s * z) with log-scales
lowered by ln 1.6; new Gaussians after the kept ones, with zero moments.  Checked against
numpy indexing, scipy's quaternion rotation and hand-built edge cases.
"""
import math

import numpy as np
import pytest
from scipy.spatial.transform import Rotation

import oracle


def _scene(n, seed):
    rng = np.random.default_rng(seed)
    P = rng.normal(size=(15, n, 4)).astype(np.float32)
    P[1, :, :3] = rng.uniform(-4.0, -1.0, size=(n, 3))
    P[1, :, 3] = 0.0
    M = rng.normal(size=(15, n, 4)).astype(np.float32)
    V = np.abs(rng.normal(size=(15, n, 4))).astype(np.float32)
    Z = rng.standard_normal((n, 6)).astype(np.float32)
    return P, M, V, Z


def _expected(P, M, V, stat, thr, lthr, Z):
    """The same output from numpy and scipy, written independently."""
    n = P.shape[1]
    cnt = stat[:, 1]
    with np.errstate(divide="ignore", invalid="ignore"):
        avg = np.where(cnt > 0, stat[:, 0] / np.where(cnt > 0, cnt, 1), 0).astype(np.float32)
    sel = (cnt > 0) & (avg >= np.float32(thr))
    big = P[1, :, :3].max(axis=1) > np.float32(lthr)
    split, clone = sel & big, sel & ~big
    keep = ~split
    outs_p = [P[:, keep].astype(np.float64)]
    outs_m = [M[:, keep].astype(np.float64)]
    outs_v = [V[:, keep].astype(np.float64)]
    for i in np.nonzero(sel)[0]:
        if clone[i]:
            outs_p.append(P[:, i:i + 1].astype(np.float64))
            outs_m.append(np.zeros((15, 1, 4)))
            outs_v.append(np.zeros((15, 1, 4)))
            continue
        w, x, y, z = P[2, i].astype(np.float64)
        R = Rotation.from_quat([x, y, z, w]).as_matrix()
        s = np.exp(P[1, i, :3].astype(np.float64))
        for k in range(2):
            c = P[:, i:i + 1].astype(np.float64).copy()
            c[0, 0, :3] += R @ (s * Z[i, 3 * k:3 * k + 3].astype(np.float64))
            c[1, 0, :3] -= math.log(1.6)
            outs_p.append(c)
            outs_m.append(np.zeros((15, 1, 4)))
            outs_v.append(np.zeros((15, 1, 4)))
    cat = lambda xs: np.concatenate(xs, axis=1)
    return cat(outs_p), cat(outs_m), cat(outs_v), int(clone.sum()), int(split.sum())


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_densify_matches_numpy_and_scipy(seed):
    n = 300
    P, M, V, Z = _scene(n, seed)
    rng = np.random.default_rng(100 + seed)
    stat = np.zeros((n, 2), np.float32)
    stat[:, 1] = rng.integers(0, 5, size=n)
    stat[:, 0] = rng.uniform(0, 2e-3, size=n) * stat[:, 1]
    thr, lthr = 2e-4 * 4, -2.5
    (op, om, ov), (nc, ns) = oracle.densify(P, M, V, stat, thr, lthr, Z)
    ep, em, ev, enc, ens = _expected(P, M, V, stat, thr, lthr, Z)
    assert (nc, ns) == (enc, ens)
    assert nc > 10 and ns > 10 and (stat[:, 1] == 0).sum() > 10  # every branch is exercised
    assert op.shape == ep.shape == (15, n + nc + ns, 4)
    assert np.allclose(op, ep, rtol=1e-12, atol=1e-12)
    assert (om == em).all() and (ov == ev).all()


def test_densify_edges():
    """A mean exactly at the threshold is selected (>=), a largest log-scale exactly at its
    threshold clones (>), a Gaussian never seen is never selected, nothing selected leaves
    the model as it was."""
    n = 4
    P, M, V, Z = _scene(n, 7)
    P[1, :, :3] = -3.0
    P[1, 1, 2] = -2.0  # largest log-scale exactly at the threshold below
    P[1, 2, 0] = -1.5  # above it
    stat = np.array([[0.5, 2.0], [0.75, 3.0], [0.25, 1.0], [9.0, 0.0]], np.float32)  # means .25, .25, .25, -
    (op, om, ov), (nc, ns) = oracle.densify(P, M, V, stat, 0.25, -2.0, Z)
    assert (nc, ns) == (2, 1)  # 0 and 1 cloned, 2 split, 3 never seen
    assert op.shape[1] == 4 - 1 + 2 + 2
    assert np.array_equal(op[:, :3], P[:, [0, 1, 3]].astype(np.float64))
    assert np.array_equal(op[:, 3], P[:, 0].astype(np.float64)) and np.array_equal(op[:, 4], P[:, 1].astype(np.float64))
    assert (om[:, 3:] == 0).all() and (ov[:, 3:] == 0).all()
    assert np.array_equal(om[:, :3], M[:, [0, 1, 3]].astype(np.float64))
    # the split children straddle the parent along its rotated, scaled axes
    c0, c1 = op[0, 5, :3], op[0, 6, :3]
    assert not np.allclose(c0, P[0, 2, :3]) and np.allclose(op[1, 5, :3], P[1, 2, :3] - math.log(1.6))
    (op2, _, _), (nc2, ns2) = oracle.densify(P, M, V, stat, 10.0, -2.0, Z)
    assert (nc2, ns2) == (0, 0) and np.array_equal(op2, P.astype(np.float64))


def test_densify_statistic():
    rng = np.random.default_rng(3)
    n = 50
    g2d = rng.normal(size=(n, 9))
    radius = np.where(rng.uniform(size=n) < 0.6, 3, 0).astype(np.int32)
    stat = oracle.densify_stat(g2d, radius)
    stat = oracle.densify_stat(2 * g2d, radius, stat)  # a second view, twice the gradient
    want = 3 * np.hypot(g2d[:, 0], g2d[:, 1]) * (radius > 0)
    assert np.allclose(stat[:, 0], want, rtol=1e-14)
    assert np.array_equal(stat[:, 1], 2.0 * (radius > 0))
