"""Parity at the full sizes of the five workloads (GB300 only).

Stage-wise: the CUDA stages receive the oracle's own projection (cast to fp32) so every later
stage is compared on identical inputs.  Where the oracle cannot finish a whole view in
seconds, the comparison is restricted to sampled tiles (bit-exact lists, composited pixels,
screen-space gradients of the Gaussians in them) and sampled Gaussians (projection,
projection backward, Adam); set sizes and overlaps are exact at any size.

Whole step: the trainer's own path (batched projection, batched sorts, compositing, loss,
compositing backward, fused projection backward + Adam) runs at full size from the
parameters alone, and the oracle recomputes sampled Gaussians of every view of the batch
from crops around them (tests/sampled_step.py).
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import scenes  # noqa: E402
from gaussian_splatting_gb300 import _native as N  # noqa: E402
from gaussian_splatting_gb300.trainer import Trainer  # noqa: E402

from parity import (FLAG_FRAC_GAUSSIANS, FLAG_FRAC_PIXELS, FLAG_FRAC_VALUES, IMG_ATOL, MARGIN, RTOL, ATOL, allclose_grad,  # noqa: E402
                    dev, flag_img_bound, grad2d_oracle_layout, host, oracle_inputs_from_planes,
                    proj_planes_from_oracle, report)
from sampled_step import pick_sample, sampled_step  # noqa: E402

pytestmark = pytest.mark.gpu

_SCENES = {}


def scene_params(cfg):
    """Parameters of a workload, generated once per test session (the 40M scene is 9.6 GB)."""
    if cfg not in _SCENES:
        _SCENES[cfg] = scenes.make_params(cfg)
    return _SCENES[cfg]


def project_chunked(P, cam, chunk=2_000_000):
    """Oracle projection of every Gaussian, in column chunks to bound host memory."""
    n = P.shape[1]
    out = {k: [] for k in ("uvzo", "conic", "radius", "rgb", "tiles", "margin")}
    for a in range(0, n, chunk):
        pr = oracle.project(P[:, a:a + chunk], cam)
        for k in out:
            out[k].append(pr[k].astype(np.float32) if pr[k].dtype == np.float64 and k != "margin" else pr[k])
    return {k: np.concatenate(v) for k, v in out.items()}


def tile_lists_oracle(planes, cam, tiles):
    """Depth-sorted Gaussian list of each sampled tile from the fp32 stage inputs
    (rectangle test + stable order by (fp32 depth, index))."""
    u = planes[0, :, 0].astype(np.float64)
    v = planes[0, :, 1].astype(np.float64)
    z = planes[0, :, 2]
    r = planes[1, :, 3].view(np.int32).astype(np.int64)
    fu, fv = np.floor(u).astype(np.int64), np.floor(v).astype(np.int64)
    x0 = np.clip((fu - r) // 16, 0, cam.tiles_x)
    x1 = np.clip((fu + r) // 16 + 1, 0, cam.tiles_x)
    y0 = np.clip((fv - r) // 16, 0, cam.tiles_y)
    y1 = np.clip((fv + r) // 16 + 1, 0, cam.tiles_y)
    out = {}
    for t in tiles:
        tx, ty = t % cam.tiles_x, t // cam.tiles_x
        sel = np.nonzero((r > 0) & (x0 <= tx) & (tx < x1) & (y0 <= ty) & (ty < y1))[0]
        order = np.lexsort((sel, z[sel].view(np.uint32)))
        out[t] = sel[order].astype(np.uint32)
    return out


def gpu_bin(planes, cam):
    n = planes.shape[1]
    capacity = int(planes[2, :, 3].view(np.int32).astype(np.int64).sum()) + 1
    ws_b = N.gs_bin_sort_workspace_size(n, capacity, cam)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    keys = torch.empty(capacity, dtype=torch.int64, device="cuda")
    vals = torch.empty(capacity, dtype=torch.int32, device="cuda")
    ranges = torch.zeros((cam.tiles_x * cam.tiles_y, 2), dtype=torch.int32, device="cuda")
    count = torch.zeros(2, dtype=torch.int64, device="cuda")
    dp = dev(planes)
    M = N.gs_bin_sort(dp, n, cam, ws, ws_b, keys, vals, capacity, ranges, count, sync=True)
    return dp, keys, vals, ranges, M


@pytest.mark.parametrize("cfg,view", [(2, 0), (2, 3), (3, 0), (4, 5)])
def test_sampled_tiles_at_full_size(cfg, view):
    P = scene_params(cfg)
    cam = scenes.make_cameras(cfg)[view]
    n = P.shape[1]
    pr = project_chunked(P, cam)
    planes = proj_planes_from_oracle(pr)
    del pr
    # projection on a sample of Gaussians
    rng = np.random.default_rng(cfg * 100 + view)
    idx = np.sort(rng.choice(n, 100_000, replace=False))
    proj = torch.zeros((3, n, 4), dtype=torch.float32, device="cuda")
    Pd = dev(P)
    N.gs_project(Pd, n, cam, proj)
    torch.cuda.synchronize()
    g = host(proj[:, torch.from_numpy(idx).cuda()])
    pr_s = oracle.project(P[:, idx], cam)
    ok = pr_s["margin"] >= MARGIN
    okv = ok & (pr_s["rmargin"] >= MARGIN)
    report(f"cfg{cfg} view{view} projection: flagged decisions", int((~ok).sum()), len(idx))
    report(f"cfg{cfg} view{view} projection: flagged radius / rectangle values", int((~okv).sum()), len(idx))
    assert (~ok).sum() <= max(2, FLAG_FRAC_GAUSSIANS * len(idx))
    assert (~okv).sum() <= max(2, FLAG_FRAC_VALUES * len(idx))
    assert np.array_equal(g[1, okv, 3].view(np.int32), pr_s["radius"][okv])
    del proj, Pd
    # binning: bit-exact lists of sampled tiles (on the oracle's projection)
    dp, keys, vals, ranges, M = gpu_bin(planes, cam)
    rg = host(ranges).view(np.uint32)
    lens = rg[:, 1] - rg[:, 0]
    busy = np.nonzero(lens)[0]
    assert busy.size > 0
    tiles = list(rng.choice(busy, min(10, busy.size), replace=False)) + [int(np.argmax(lens))]
    want = tile_lists_oracle(planes, cam, tiles)
    vh = host(vals).view(np.uint32)
    kh = host(keys).view(np.uint64)
    assert M == int(planes[2, :, 3].view(np.int32).astype(np.int64).sum())
    for t in tiles:
        got = vh[rg[t, 0]:rg[t, 1]]
        assert np.array_equal(got, want[t]), t
        exp_keys = (np.uint64(t) << np.uint64(32)) | planes[0, got, 2].view(np.uint32).astype(np.uint64)
        assert np.array_equal(kh[rg[t, 0]:rg[t, 1]], exp_keys)
    # compositing on the sampled tiles only (both sides see only their lists)
    mini_ranges = np.zeros_like(rg)
    mini_vals = []
    off = 0
    for t in tiles:
        mini_vals.append(want[t])
        mini_ranges[t] = (off, off + len(want[t]))
        off += len(want[t])
    mini_vals = np.concatenate(mini_vals).astype(np.uint32)
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    img_o, T_o, nc_o, mg = oracle.render_fwd(uvzo, conic, rgb, mini_vals, mini_ranges, cam.width, cam.height)
    H, W = cam.height, cam.width
    img = torch.zeros((3, H, W), device="cuda")
    T = torch.zeros((H, W), device="cuda")
    nc = torch.zeros((H, W), dtype=torch.int32, device="cuda")
    mv, mr = dev(mini_vals.view(np.int32)), dev(mini_ranges.view(np.int32))
    N.gs_render_fwd(dp, n, mv, mr, cam, None, img, T, nc)
    torch.cuda.synchronize()
    img_h, T_h, nc_h = host(img), host(T), host(nc).view(np.uint32)
    okp = mg >= MARGIN
    report(f"cfg{cfg} view{view} flagged pixels", int((~okp).sum()), okp.size)
    # (a floor of 8 for a sample of a few thousand pixels that always holds the view's busiest
    # tile, whose pixels carry thousands of decisions each)
    assert (~okp).sum() <= max(8, FLAG_FRAC_PIXELS * 256 * len(tiles))
    assert np.abs(img_h - img_o)[:, okp].max() <= IMG_ATOL
    assert np.array_equal(nc_h[okp], nc_o[okp])
    if (~okp).any():
        assert np.abs(img_h - img_o)[:, ~okp].max() <= flag_img_bound(rgb)
    # compositing backward on the same tiles, with a gradient nonzero only there and zero on
    # the pixels whose decisions sit on a threshold (on both sides: nothing is set aside)
    dimg = np.zeros((3, H, W), np.float32)
    for t in tiles:
        tx, ty = t % cam.tiles_x, t // cam.tiles_x
        dimg[:, ty * 16:ty * 16 + 16, tx * 16:tx * 16 + 16] = rng.normal(0, 1e-4, size=(3, 16, 16)).astype(np.float32)[
            :, : min(16, H - ty * 16), : min(16, W - tx * 16)]
    dimg *= okp[None]
    g_o = oracle.render_bwd(uvzo, conic, rgb, mini_vals, mini_ranges, W, H, dimg.astype(np.float64))
    grad2d = torch.zeros((n, 12), device="cuda")
    N.gs_render_bwd(dp, n, mv, mr, cam, None, dev(T_o.astype(np.float32)), dev(nc_o.view(np.int32)), dev(dimg), grad2d)
    torch.cuda.synchronize()
    members = np.unique(mini_vals)
    gm = grad2d_oracle_layout(host(grad2d[torch.from_numpy(members.astype(np.int64)).cuda()]))
    bad = allclose_grad(gm, g_o[members])
    report(f"cfg{cfg} view{view} render_bwd (every Gaussian of the tiles)", int(bad.sum()), bad.size)
    assert bad.sum() == 0


@pytest.mark.parametrize("cfg", [3, 4])
def test_projection_backward_and_adam_on_sampled_gaussians(cfg):
    P = scene_params(cfg)
    cam = scenes.make_cameras(cfg)[1]
    n = P.shape[1]
    rng = np.random.default_rng(cfg)
    idx = np.sort(rng.choice(n, 50_000, replace=False))
    # projection backward on the full arrays, gradient planted on the sampled Gaussians
    pr_s = oracle.project(P[:, idx], cam)
    ok = (pr_s["margin"] >= MARGIN) & ((np.abs(pr_s["raw"]) > 1e-4).all(axis=1) | (pr_s["radius"] == 0))
    g2d_s = rng.normal(0, 1e-3, size=(len(idx), 9)) * ((pr_s["radius"] > 0) & ok)[:, None]
    g2d_s = g2d_s.astype(np.float32).astype(np.float64)
    ref = oracle.project_bwd(P[:, idx], cam, g2d_s)
    planes = np.zeros((3, n, 4), np.float32)
    planes_s = proj_planes_from_oracle(pr_s)
    planes[:, idx] = planes_s
    g2d = np.zeros((n, 12), np.float32)
    g2d[idx[:, None], np.array([0, 1, 4, 5, 6, 2, 8, 9, 10])[None, :]] = g2d_s
    grads = torch.zeros((15, n, 4), device="cuda")
    N.gs_project_bwd(dev(P), n, cam, dev(planes), dev(g2d), grads)
    torch.cuda.synchronize()
    got = host(grads[:, torch.from_numpy(idx).cuda()]).astype(np.float64)
    bad = allclose_grad(got, ref)
    bad[1, :, 3] = False
    report(f"cfg{cfg} project_bwd sample", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    del grads
    # Adam on the whole model with a union list, checked on the sampled rows
    G = rng.normal(0, 1e-3, size=(15, len(idx), 4)).astype(np.float32)
    union = np.sort(rng.choice(n, n // 3, replace=False)).astype(np.uint32)
    uset = np.isin(idx, union)
    tp, tg = dev(P), torch.zeros((15, n, 4), device="cuda")
    tg[:, torch.from_numpy(idx).cuda()] = dev(G)
    tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
    nu = torch.tensor([len(union)], dtype=torch.int64, device="cuda")
    N.gs_sparse_adam(tp, tg, tm, tv, n, dev(union.view(np.int32)), nu, n, 1e-3, 0.9, 0.999, 1e-15, 4, 3)
    torch.cuda.synchronize()
    sel = torch.from_numpy(idx).cuda()
    p_new, m_new = host(tp[:, sel]), host(tm[:, sel])
    rows = np.nonzero(uset)[0]
    ref_p, _, ref_m, _ = oracle.sparse_adam(P[:, idx], G, np.zeros_like(G), np.zeros_like(G), rows.astype(np.uint32),
                                            1e-3, 0.9, 0.999, 1e-15, 4, 3)
    assert allclose_grad(p_new, ref_p).sum() == 0
    assert allclose_grad(m_new, ref_m).sum() == 0
    assert (p_new[:, ~uset] == P[:, idx][:, ~uset]).all()


def test_visible_sets_sixteen_views_at_forty_million():
    B, n = 16, 40_000_000
    rng = np.random.default_rng(44)
    projs, bits = [], []
    for b in range(B):
        vis = rng.uniform(size=n) < (0.05 + 0.05 * b)
        radii = np.where(vis, 3, 0).astype(np.int32)
        q = torch.zeros((3, n, 4), dtype=torch.float32, device="cuda")
        q[1, :, 3] = dev(radii.view(np.float32))
        projs.append(q)
        bits.append(vis)
    ws_b = N.gs_visible_sets_workspace_size(B, n)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    off = torch.zeros(B + 1, dtype=torch.int64, device="cuda")
    ind = torch.zeros(B * n, dtype=torch.int32, device="cuda")
    uni = torch.zeros(n, dtype=torch.int32, device="cuda")
    nu = torch.zeros(1, dtype=torch.int64, device="cuda")
    inter = torch.zeros((B, B), dtype=torch.int64, device="cuda")
    jac = torch.zeros((B, B), dtype=torch.float32, device="cuda")
    N.gs_visible_sets(projs, B, n, ws, ws_b, off, ind, uni, nu, inter, jac)
    torch.cuda.synchronize()
    counts = np.array([b.sum() for b in bits])
    assert np.array_equal(np.diff(host(off)), counts)
    for b in (0, 7, 15):  # ascending lists, spot-checked views
        lo, hi = host(off)[b], host(off)[b + 1]
        assert np.array_equal(host(ind[lo:hi]).view(np.uint32), np.nonzero(bits[b])[0].astype(np.uint32))
    un = np.logical_or.reduce(bits)
    assert int(nu.item()) == un.sum()
    assert np.array_equal(host(uni[: un.sum()]).view(np.uint32), np.nonzero(un)[0].astype(np.uint32))
    ih, jh = host(inter), host(jac)
    for i in range(B):
        for j in range(i, B):
            c = int(np.count_nonzero(bits[i] & bits[j]))
            assert ih[i, j] == c and ih[j, i] == c
            u = counts[i] + counts[j] - c
            assert jh[i, j] == np.float32(c / u)


def test_render_bwd_full_image_benchmark_view():
    """Compositing backward over a whole 1236x820 view of the 300K-Gaussian scene, every
    Gaussian compared, nothing set aside: both sides get the oracle's projection, lists and
    forward state, and the loss gradient of a jittered-scene target with the pixels whose
    compositing decisions sit on a threshold zeroed on both sides."""
    P = scenes.make_params(1)
    cam = scenes.make_cameras(1)[5]
    n = P.shape[1]
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    keys, vals, ranges = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
    img, T_o, nc_o, mg = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height)
    tgt = oracle.render_view(scenes.jitter_means(P, 0.02, 2001), cam)
    _, dimg = oracle.loss(img.astype(np.float32), tgt.astype(np.float32), scale=0.25)
    flagged = mg < MARGIN
    report("full-image render_bwd: flagged pixels (gradient zeroed)", int(flagged.sum()), flagged.size)
    assert flagged.sum() <= max(2, FLAG_FRAC_PIXELS * flagged.size)
    dimg32 = (dimg * ~flagged[None]).astype(np.float32)
    g_o = oracle.render_bwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height, dimg32.astype(np.float64))
    grad2d = torch.full((n, 12), 5.0, dtype=torch.float32, device="cuda")
    N.gs_render_bwd(dev(planes), n, dev(vals.view(np.int32)), dev(ranges.view(np.int32)), cam, None,
                    dev(T_o.astype(np.float32)), dev(nc_o.view(np.int32)), dev(dimg32), grad2d)
    torch.cuda.synchronize()
    gm = grad2d_oracle_layout(host(grad2d))
    bad = allclose_grad(gm, g_o)
    report("full-image render_bwd (every Gaussian, nothing set aside)", int(bad.sum()), bad.size)
    assert (np.abs(g_o).sum(axis=1) > 0).sum() > 20_000  # the view's Gaussians are covered
    assert bad.sum() == 0


def flagged_pixel_gradient(P, cam, pr, target, batch):
    """The oracle's parameter gradient of one view of a step restricted to the pixels whose
    compositing decisions sit within MARGIN of a threshold (the loss gradient zeroed on every
    other pixel; only the tiles holding such pixels are walked)."""
    keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], cam.width, cam.height)
    img, _, _, mg = oracle.render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, cam.width, cam.height)
    _, dimg = oracle.loss(img, target, scale=1.0 / batch)
    flagged = mg < MARGIN
    dimg *= flagged[None]
    busy = np.zeros(cam.tiles_x * cam.tiles_y, bool)
    ys, xs = np.nonzero(flagged)
    busy[(ys // 16) * cam.tiles_x + xs // 16] = True
    r2 = ranges.copy()
    r2[~busy] = 0
    g2d = oracle.render_bwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, r2, cam.width, cam.height, dimg)
    return oracle.project_bwd(P, cam, g2d)


def test_full_step_parity_at_benchmark_size():
    """One whole training step (4 views of the 300K-Gaussian, 1236x820 workload, batch 4), from
    the parameters alone, every Gaussian compared except those whose own projection decision
    (cull, radius ceiling, tile rectangle) sits on its threshold in one of the views."""
    cfg = scenes.CONFIGS[1]
    P = scenes.make_params(1)
    cams = [scenes.make_cameras(1)[v] for v in scenes.batch_views(cfg, 0)]
    jit = scenes.jitter_means(P, cfg.jitter, 2001)
    tg = np.stack([oracle.render_view(jit, c) for c in cams]).astype(np.float32)
    ref = oracle.step(P, np.zeros_like(P), np.zeros_like(P), cams, tg, lr=cfg.lr, eps=cfg.eps)
    tr = Trainer(dev(P), cfg.width, cfg.height, cfg.batch, lr=cfg.lr, eps=cfg.eps)
    res = tr.step_async(cams, dev(tg), adam=False)
    torch.cuda.synchronize()
    assert (host(res.status)[:, 1] == 0).all()
    assert float(res.loss.item()) == pytest.approx(ref["loss"], rel=1e-5)
    G = ref["grads"]
    g = host(tr.grads).astype(np.float64)
    # set aside (1) Gaussians whose own projection decision sits on its threshold in a view and
    # (2) Gaussians for which the pixels with a compositing decision on its threshold carry a
    # quarter of the gradient tolerance or more: the oracle's gradient of the step restricted
    # to those pixels (a flipped decision there changes a contribution by up to all of it)
    proj_aside = np.zeros(P.shape[1], bool)
    G_flag = np.zeros_like(G)
    for b, cam in enumerate(cams):
        pr = oracle.project(P, cam)
        proj_aside |= pr["margin"] < MARGIN
        G_flag += flagged_pixel_gradient(P, cam, pr, tg[b], len(cams))
    tol = RTOL * np.abs(G) + ATOL
    pix_aside = (np.abs(G_flag) > 0.25 * tol).any(axis=(0, 2))
    aside = proj_aside | pix_aside
    report("benchmark-size step: Gaussians set aside for their projection", int(proj_aside.sum()), aside.size)
    report("benchmark-size step: Gaussians set aside for flagged pixels", int((pix_aside & ~proj_aside).sum()),
           aside.size)
    assert aside.mean() < 1e-3
    bad = allclose_grad(g, G)
    bad[1, :, 3] = False  # padding lane
    report("benchmark-size step grads, every entry", int(bad.sum()), bad.size)
    bad = bad[:, ~aside]
    report("benchmark-size step grads outside the set-aside", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    # the batched, visible-only update (lr sqrt(4), beta^4): at t = 1 each entry moves by
    # lr' sign(g), so entries whose gradient lies within the 1e-6 floor of zero are not compared
    tr.grads.zero_()
    loss = tr.step(cams, dev(tg))
    assert loss == pytest.approx(ref["loss"], rel=1e-5)
    Pn = host(tr.params).astype(np.float64)
    clear = (np.abs(G) > 1e-6) & ~aside[None, :, None]
    bad = allclose_grad(Pn - P, ref["params"] - P, RTOL, 1e-6)[clear]
    report("benchmark-size step params", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    untouched = ~((ref["params"] != P).any(axis=(0, 2)))
    assert (Pn[:, untouched] == P[:, untouched]).all()


# the batches checked through the trainer's own path: the unbounded scene's first batch holds
# two sky views (3 and 7); the 4K scene's first batch is the full 16 views of one fused update
TRAINER_CASES = [(2, (0, 3)), (3, (0, 2)), (4, (0, 9))]


@pytest.mark.parametrize("cfg_idx,pick_views", TRAINER_CASES)
def test_trainer_step_on_sampled_gaussians_at_full_size(cfg_idx, pick_views):
    """The trainer's whole step at full size (batched projection and sorts, per-view
    compositing, loss and backward, the fused projection backward + Adam over the batch)
    against the oracle on sampled Gaussians: per-view screen-space gradients, the summed
    parameter gradients and the updated parameters."""
    cfg = scenes.CONFIGS[cfg_idx]
    P = scene_params(cfg_idx)
    cams = [scenes.make_cameras(cfg_idx)[v] for v in scenes.batch_views(cfg, 0)]
    B = len(cams)
    tg = scenes.synthetic_targets(B, cfg.width, cfg.height, 3000 + cfg_idx)
    rmax = 24 if cfg.width > 2000 else 12
    sample = np.union1d(pick_sample(P, cams[pick_views[0]], 8, 10 + cfg_idx, rmax),
                        pick_sample(P, cams[pick_views[1]], 8, 20 + cfg_idx, rmax))
    workers = max(1, min(16, len(os.sched_getaffinity(0))))  # one view per host core at a time
    ref = sampled_step(P, cams, tg, sample, lr=cfg.lr, eps=cfg.eps, workers=workers)
    # set aside sampled Gaussians with a projection decision on its threshold in a view, or
    # whose pixels with a compositing decision on its threshold carry a quarter of a tolerance
    ok = (ref["margin"] >= MARGIN).all(axis=0)
    ok &= ~(np.abs(ref["grads_flag"]) > 0.25 * (RTOL * np.abs(ref["grads"]) + ATOL)).any(axis=(0, 2))
    ok &= ~(np.abs(ref["g2d_flag"]) > 0.25 * (RTOL * np.abs(ref["g2d"]) + ATOL)).any(axis=(0, 2))
    report(f"cfg{cfg_idx} trainer step: sampled Gaussians set aside", int((~ok).sum()), ok.size)
    assert ok.sum() >= 12
    assert ref["visible"].sum() >= 2 * B  # the sample is seen across the batch
    tr = Trainer(dev(P), cfg.width, cfg.height, B, lr=cfg.lr, eps=cfg.eps, keep_views=True)
    res = tr.step_async(cams, dev(tg), adam=False)
    torch.cuda.synchronize()
    assert (host(res.status)[:, 1] == 0).all()
    sel = torch.from_numpy(sample.astype(np.int64)).cuda()
    for b in range(B):
        g2 = grad2d_oracle_layout(host(tr.grad2d[b][sel]).astype(np.float64))
        bad = allclose_grad(g2, ref["g2d"][b])[ok]
        assert bad.sum() == 0, (b, np.abs(g2 - ref["g2d"][b])[ok].max())
    g = host(tr.grads[:, sel]).astype(np.float64)
    bad = allclose_grad(g, ref["grads"])[:, ok]
    bad[1, :, 3] = False
    report(f"cfg{cfg_idx} trainer step grads (sampled)", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    del tr
    torch.cuda.empty_cache()
    # the update through the fused projection backward + Adam (t = 1, zero moments)
    tr = Trainer(dev(P), cfg.width, cfg.height, B, lr=cfg.lr, eps=cfg.eps)
    tr.step(cams, dev(tg))
    Pn = host(tr.params[:, sel]).astype(np.float64)
    P0 = P[:, sample].astype(np.float64)
    clear = (np.abs(ref["grads"]) > 1e-6) & ok[None, :, None]
    bad = allclose_grad(Pn - P0, ref["params"] - P0, RTOL, 1e-6)[clear]
    report(f"cfg{cfg_idx} trainer step params (sampled)", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    unseen = ~ref["visible"].any(axis=0)
    assert (Pn[:, unseen] == P0[:, unseen]).all()
    del tr
    torch.cuda.empty_cache()
