"""The sampled full-size step (tests/sampled_step.py) reproduces the oracle's whole step.

On a scene small enough for oracle.step, the per-view screen-space gradients, the summed
parameter gradients and the Adam update of sampled Gaussians, computed from crops around each
Gaussian's tile rectangle, equal those of the whole step up to summation order.  The sample
includes a Gaussian that only the second view sees.  A second test plants mistakes in copies
of sampled_step.py and checks that this comparison fails on each.
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
    only_second = np.zeros(0, np.int64)
    if layout_cfg == 2:
        # a Gaussian only the second view sees: the update set is the union of the views' sets
        pr0, pr1 = (oracle.project(P, c) for c in cams)
        clear = (pr0["margin"] >= 1e-4) & (pr1["margin"] >= 1e-4) & (np.abs(pr1["raw"]) > 1e-3).all(axis=1)
        only_second = np.nonzero((pr0["radius"] == 0) & (pr1["radius"] >= 2) & (pr1["radius"] <= 14) & clear)[0][:1]
        assert only_second.size == 1
        sample = np.union1d(sample, only_second)
    assert sample.size >= 8
    got = sampled_step(P, cams, tg, sample, lr=cfg.lr, eps=cfg.eps, workers=2 if layout_cfg == 2 else 1)
    for b in range(len(cams)):
        ref = g2d_whole[b][sample]
        assert np.allclose(got["g2d"][b], ref, rtol=1e-9, atol=1e-15 * max(1.0, np.abs(ref).max()))
    assert np.allclose(got["grads"], whole["grads"][:, sample], rtol=1e-9, atol=1e-18)
    assert np.allclose(got["params"], whole["params"][:, sample], rtol=1e-12, atol=1e-15)
    # the sample is not trivial: its Gaussians have gradients in both views
    assert (np.abs(got["g2d"]).sum(axis=2) > 0).sum() >= 8
    for i in only_second:
        k = int(np.nonzero(sample == i)[0][0])
        assert not got["visible"][0, k] and got["visible"][1, k]
        assert (got["params"][:, k] != P[:, i]).any()  # updated through the second view alone


# mistakes planted in copies of sampled_step.py: (text occurring once, replacement).  Not among
# them, as they change no result: widening the region whose loss gradient is kept to the
# grown crop (the sampled Gaussian has no pixel outside its own tiles), and trimming the reach
# bound's slack (the bound already rounds out to whole tiles).
SAMPLED_MUTATIONS = {
    # the crop not grown by a ring of tiles (the loss gradient near its edge is then wrong)
    "no_ring": ('outer = {k: tile_box(pr_s["rect"][k], cam, 1) for k in vis}',
                'outer = {k: tile_box(pr_s["rect"][k], cam, 0) for k in vis}'),
    # the loss normalised by the crop's pixels instead of the whole image's
    "scale_by_crop": ("scale = (1.0 / batch) * (cw * ch) / (W * H)", "scale = 1.0 / batch"),
    # tile lists ordered by index instead of (depth, index)
    "order_by_index": ("sel = sel[np.lexsort((cand[live[inbox[sel]]], zb[inbox[sel]]))]",
                       "sel = sel[np.lexsort((zb[inbox[sel]], cand[live[inbox[sel]]]))]"),
    # Adam without the batch scaling
    "adam_unbatched": ("np.zeros_like(Ps, dtype=np.float64), union, lr, beta1, beta2, eps, B, step)",
                       "np.zeros_like(Ps, dtype=np.float64), union, lr, beta1, beta2, eps, 1, step)"),
    # the views' parameter gradients not summed
    "grads_last_view": ('out["grads"] += oracle.project_bwd(Ps, cam, g2d)',
                        'out["grads"] = oracle.project_bwd(Ps, cam, g2d)'),
    # the update set taken from the first view
    "union_first_view": ('union = np.nonzero(out["visible"].any(axis=0))[0].astype(np.uint32)',
                         'union = np.nonzero(out["visible"][0])[0].astype(np.uint32)'),
}


def _run_with(module_text):
    """The equality test above, in a child process that imports the given sampled_step source
    ahead of the real one."""
    import os
    import subprocess
    import sys
    import tempfile

    here = os.path.dirname(os.path.abspath(__file__))
    with tempfile.TemporaryDirectory() as d:
        with open(os.path.join(d, "sampled_step.py"), "w") as fh:
            fh.write(module_text)
        env = dict(os.environ, PYTHONPATH=d)
        cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "--import-mode=append",
               os.path.join(here, "test_oracle_sampled.py") + "::test_sampled_step_equals_whole_step"]
        r = subprocess.run(cmd, cwd=os.path.dirname(here), env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-2000:] + r.stderr[-500:]


def test_planted_mistakes_in_the_sampled_step_fail_the_comparison():
    import concurrent.futures
    import os

    src_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "sampled_step.py")
    text = open(src_path).read()
    for name, (old, _) in SAMPLED_MUTATIONS.items():
        assert text.count(old) == 1, name
    jobs = {None: text.replace('"""Oracle side', '"""(copy) Oracle side', 1)}
    jobs.update({name: text.replace(old, new) for name, (old, new) in SAMPLED_MUTATIONS.items()})
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(2, min(len(jobs), os.cpu_count() or 2))) as ex:
        res = dict(zip(jobs, ex.map(_run_with, jobs.values())))
    rc, out = res.pop(None)
    assert rc == 0, "the unmutated copy fails:\n" + out  # the copy is the one imported
    survived = {name: out for name, (rc, out) in res.items() if rc == 0 or "failed" not in out}
    assert not survived, survived
