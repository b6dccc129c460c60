"""The sampled full-size step (tests/sampled_step.py) reproduces the oracle's whole step.

On a scene small enough for oracle.step, the per-view screen-space gradients, the summed
parameter gradients and the Adam update of sampled Gaussians, computed from crops around each
Gaussian's tile rectangle, equal those of the whole step up to summation order.
"""
import numpy as np
import pytest

import oracle
import scenes
from sampled_step import pick_sample, sampled_step


@pytest.mark.parametrize("layout_cfg,seed", [(1, 3), (2, 4)])
def test_sampled_step_equals_whole_step(layout_cfg, seed):
    cfg = scenes.CONFIGS[layout_cfg]
    P = scenes.make_params(layout_cfg, seed=seed, n=12_000)
    # same camera placement at a reduced image size (and focal), two views incl. a ragged edge
    W, H, f = 200, 136, 180.0
    cams = []
    for v in (0, 3):
        c = scenes.make_cameras(layout_cfg)[v]
        cams.append(scenes.Camera(c.R, c.t, f, f, W / 2.0, H / 2.0, c.znear, W, H))
    tg = scenes.synthetic_targets(len(cams), W, H, seed)
    whole = oracle.step(P, np.zeros_like(P), np.zeros_like(P), cams, tg, lr=cfg.lr, eps=cfg.eps)
    # per-view screen-space gradients of the whole step
    g2d_whole = []
    for b, cam in enumerate(cams):
        pr = oracle.project(P, cam)
        keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], W, H)
        img, _, _, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, W, H)
        _, d = oracle.loss(img, tg[b], scale=1.0 / len(cams))
        g2d_whole.append(oracle.render_bwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, W, H, d))
    sample = np.union1d(pick_sample(P, cams[0], 6, seed, rmax=14), pick_sample(P, cams[1], 6, seed + 1, rmax=14))
    assert sample.size >= 8
    got = sampled_step(P, cams, tg, sample, lr=cfg.lr, eps=cfg.eps, workers=2 if layout_cfg == 2 else 1)
    for b in range(len(cams)):
        ref = g2d_whole[b][sample]
        assert np.allclose(got["g2d"][b], ref, rtol=1e-9, atol=1e-15 * max(1.0, np.abs(ref).max()))
    assert np.allclose(got["grads"], whole["grads"][:, sample], rtol=1e-9, atol=1e-18)
    assert np.allclose(got["params"], whole["params"][:, sample], rtol=1e-12, atol=1e-15)
    # the sample is not trivial: its Gaussians have gradients in both views
    assert (np.abs(got["g2d"]).sum(axis=2) > 0).sum() >= 8
