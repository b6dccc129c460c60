"""The synthetic workloads have the properties their descriptions give them.

The two city workloads (11M Gaussians at 1920x1080, 40M at 3840x2160) are drawn so that at
least 90 % of the projected radii stay below 2 % of the image width (the observation the
pages make about trained scenes: most Gaussians are small, which keeps the per-pixel lists
short).  The check projects a sample of each layout with the oracle from four views around
the orbit; the draws are per-Gaussian independent given the layout, so a 50,000-Gaussian draw
of the same layout has the same radius distribution as the full scene.
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
