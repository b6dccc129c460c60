"""The synthetic workloads have the properties their descriptions give them.

The two city workloads (11M Gaussians at 1920x1080, 40M at 3840x2160) are drawn so that at
least 90 % of the projected radii stay below 2 % of the image width (the observation the
pages make about trained scenes: most Gaussians are small, which keeps the per-pixel lists
short).  The check projects a sample of each layout with the oracle from four views around
the orbit; the draws are per-Gaussian independent given the layout, so a 50,000-Gaussian draw
of the same layout has the same radius distribution as the full scene.

The recipes themselves are checked too: the parameter distributions every layout shares, each
layout's structure (a cube, 64 clusters inside radius 2, a core of radius 1.5 with a
log-uniform shell to 50, 16 x 16 and 32 x 32 city blocks), and each workload's camera rig,
image size, focal length, view count, batch and Gaussian count.
"""
import numpy as np
import pytest

import oracle
import scenes


@pytest.mark.parametrize("cfg_idx", [3, 4])
def test_city_footprints_mostly_below_two_percent_of_width(cfg_idx):
    cfg = scenes.CONFIGS[cfg_idx]
    P = scenes.make_params(cfg_idx, n=50_000)
    cams = scenes.make_cameras(cfg_idx)
    for v in (0, 16, 32, 48):
        pr = oracle.project(P, cams[v])
        r = pr["radius"][pr["radius"] > 0]
        assert r.size > 20_000  # most of the city is in view
        frac = float((r < 0.02 * cfg.width).mean())
        print(f"[workload] {cfg.name} view {v}: {frac:.4f} of {r.size} radii below 2 % of the width "
              f"(p90 {np.percentile(r, 90):.0f} px)")
        assert frac >= 0.9


def test_sky_views_look_above_the_core():
    """Every fourth view of the unbounded scene aims above the dense core, so its upper half
    sees only the sparse shell: far fewer Gaussians project there than in a level view."""
    P = scenes.make_params(2, n=60_000)
    cams = scenes.make_cameras(2)
    counts = []
    for v in (2, 3):
        pr = oracle.project(P, cams[v])
        vis = pr["radius"] > 0
        top = vis & (pr["uvzo"][:, 1] < cams[v].height / 2)
        counts.append(int(top.sum()))
    assert counts[1] < 0.5 * counts[0], counts


# ------------------------------------------------------------------ the recipes themselves
def test_parameter_distributions():
    """Every layout draws the same per-Gaussian parameters: log-scales U[-4.5, -2.5], unit
    quaternions from N(0, I4), opacity logits N(0, 1), SH DC N(0.5, 0.2), the other 45 SH
    coefficients N(0, 0.05)."""
    P = scenes.make_params(1, n=200_000)
    ls = P[1, :, :3]
    assert ls.min() >= -4.5 and ls.max() <= -2.5 and abs(ls.mean() + 3.5) < 0.01
    assert np.allclose(np.linalg.norm(P[2], axis=1), 1.0, atol=1e-6)
    assert (P[1, :, 3] == 0).all()
    logit = P[0, :, 3]
    assert abs(logit.mean()) < 0.01 and abs(logit.std() - 1.0) < 0.01
    sh = P[3:].transpose(1, 0, 2).reshape(-1, 48)
    assert abs(sh[:, :3].mean() - 0.5) < 0.002 and abs(sh[:, :3].std() - 0.2) < 0.002
    assert abs(sh[:, 3:].mean()) < 0.001 and abs(sh[:, 3:].std() - 0.05) < 0.001


def test_layouts():
    cube = scenes.make_params(0)[0, :, :3]
    assert cube.shape == (2048, 3) and cube.min() >= -1 and cube.max() <= 1
    # 64 anisotropic clusters inside radius 2: means are much closer to each other than a
    # uniform draw in the same ball would be
    cl = scenes.make_params(1, n=20_000)[0, :, :3].astype(np.float64)
    assert np.linalg.norm(cl, axis=1).max() <= 2.0 + 1e-6
    d_nn = np.sort(np.linalg.norm(cl[:500, None] - cl[None, :], axis=2), axis=1)[:, 1]
    u = np.random.default_rng(0).standard_normal((20_000, 3))
    u *= (2.0 * np.random.default_rng(1).uniform(size=(20_000, 1)) ** (1 / 3)) / np.linalg.norm(u, axis=1, keepdims=True)
    d_u = np.sort(np.linalg.norm(u[:500, None] - u[None, :], axis=2), axis=1)[:, 1]
    assert np.median(d_nn) < 0.7 * np.median(d_u)
    # unbounded: 80 % in a core of radius 1.5, the rest log-uniform out to radius 50
    r = np.linalg.norm(scenes.make_params(2, n=100_000)[0, :, :3].astype(np.float64), axis=1)
    assert abs((r <= 1.5 + 1e-6).mean() - 0.8) < 1e-3 and r.max() <= 50.0 * (1 + 1e-6)
    shell = np.log(r[r > 1.5 + 1e-6])
    assert abs(np.median(shell) - 0.5 * (np.log(1.5) + np.log(50.0))) < 0.05
    # cities: 16 x 16 and 32 x 32 box-shaped blocks on a 1.5 pitch, each 1 wide and at most 3 high
    for cfg_idx, g in ((3, 16), (4, 32)):
        m = scenes.make_params(cfg_idx, n=100_000)[0, :, :3].astype(np.float64)
        cx = np.round(m[:, 0] / 1.5 + (g - 1) / 2.0)
        cz = np.round(m[:, 2] / 1.5 + (g - 1) / 2.0)
        assert cx.min() == 0 and cx.max() == g - 1 and cz.min() == 0 and cz.max() == g - 1
        assert np.abs(m[:, 0] - (cx - (g - 1) / 2.0) * 1.5).max() <= 0.5 + 1e-6
        assert m[:, 1].max() <= 0 and m[:, 1].min() >= -3.0
        assert len(np.unique(cx * g + cz)) == g * g


def test_camera_rigs_and_sizes():
    expect = {0: (1, 128, 128, 140.0, 1), 1: (64, 1236, 820, 1100.0, 4), 2: (200, 1237, 822, 1100.0, 8),
              3: (64, 1920, 1080, 0.89 * 1920, 4), 4: (64, 3840, 2160, 0.89 * 3840, 16)}
    counts = {0: 2048, 1: 300_000, 2: 3_000_000, 3: 11_000_000, 4: 40_000_000}
    for k, (views, W, H, f, batch) in expect.items():
        cfg = scenes.CONFIGS[k]
        cams = scenes.make_cameras(k)
        assert cfg.n == counts[k] and cfg.batch == batch and len(cams) == views
        for c in cams:
            assert (c.width, c.height) == (W, H) and c.fx == c.fy == f and (c.cx, c.cy) == (W / 2, H / 2)
        centres = [-(np.asarray(c.R, np.float64).T @ np.asarray(c.t, np.float64)) for c in cams]
        if k == 0:
            assert np.allclose(centres[0], (0, 0, -4), atol=1e-6)
        if k == 1:  # a ring of radius 5 around the object
            assert np.allclose([np.linalg.norm(e) for e in centres], 5.0, atol=1e-5)
        if k == 2:  # a ring of radius 4; every fourth view aims above the core
            assert np.allclose([np.linalg.norm(e) for e in centres], 4.0, atol=1e-5)
            ups = [k2 for k2, c in enumerate(cams) if np.asarray(c.R)[2, 1] < -0.1]
            assert ups == list(range(3, 200, 4))
