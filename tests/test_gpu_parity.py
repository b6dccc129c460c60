"""Parity of every libgs.so entry point with the CPU oracle (GB300 only).

Each stage test feeds the CUDA entry point and the oracle stage the same inputs -- drawn
by the scene generator or produced by the oracle's previous stage, never by the CUDA
path -- and compares element by element under the tolerances of tests/parity.py.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import scenes  # noqa: E402
from gaussian_splatting_gb300 import _native as N  # noqa: E402
from gaussian_splatting_gb300.trainer import Trainer  # noqa: E402

from parity import (ATOL, FLAG_FRAC_GAUSSIANS, FLAG_FRAC_PIXELS, FLAG_FRAC_VALUES, IMG_ATOL, MARGIN, RTOL, allclose_grad, dev,  # noqa: E402
                    flag_img_bound, grad2d_oracle_layout, host, oracle_inputs_from_planes, proj_planes_from_oracle,
                    report)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    N.load()


def scene(cfg, n=None, view=0):
    P = scenes.make_params(cfg, n=n)
    cam = scenes.make_cameras(cfg)[view]
    return P, cam


def gpu_project(P, cam):
    n = P.shape[1]
    proj = torch.zeros((3, n, 4), dtype=torch.float32, device="cuda")
    N.gs_project(dev(P), n, cam, proj)
    torch.cuda.synchronize()
    return host(proj)


def gpu_bin_sort(planes, cam, capacity=None, with_keys=True):
    n = planes.shape[1]
    tiles = cam.tiles_x * cam.tiles_y
    if capacity is None:
        capacity = int(planes[2, :, 3].view(np.int32).astype(np.int64).sum()) + 1
    ws_bytes = N.gs_bin_sort_workspace_size(n, capacity, cam)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    keys = torch.zeros(max(capacity, 1), dtype=torch.int64, device="cuda")
    vals = torch.zeros(max(capacity, 1), dtype=torch.int32, device="cuda")
    ranges = torch.full((tiles, 2), 7, dtype=torch.int32, device="cuda")
    count = torch.zeros(2, dtype=torch.int64, device="cuda")
    M = N.gs_bin_sort(dev(planes), n, cam, ws, ws_bytes, keys if with_keys else None, vals, capacity, ranges, count,
                      sync=True)
    return (host(keys)[:M].view(np.uint64), host(vals)[:M].view(np.uint32), host(ranges).view(np.uint32), M,
            host(count))


# ------------------------------------------------------------------ projection
@pytest.mark.parametrize("cfg,n,view", [(0, None, 0), (1, 60_000, 0), (1, 60_000, 17), (2, 50_000, 3)])
def test_project_parity(cfg, n, view):
    P, cam = scene(cfg, n, view)
    g = gpu_project(P, cam)
    pr = oracle.project(P, cam)
    ok = pr["margin"] >= MARGIN            # decisions that can change an output
    okv = ok & (pr["rmargin"] >= MARGIN)   # and the integer radius / rectangle values
    rg = g[1, :, 3].view(np.int32)
    tg = g[2, :, 3].view(np.int32)
    flagged = int((~ok).sum())
    report(f"project cfg{cfg} flagged decisions", flagged, P.shape[1])
    report(f"project cfg{cfg} flagged radius / rectangle values", int((~okv).sum()), P.shape[1])
    assert flagged <= max(2, FLAG_FRAC_GAUSSIANS * P.shape[1])
    assert (~okv).sum() <= max(2, FLAG_FRAC_VALUES * P.shape[1])
    assert np.array_equal(rg[okv], pr["radius"][okv])
    assert np.array_equal(tg[okv], pr["tiles"][okv])
    assert np.array_equal(rg[ok] > 0, pr["radius"][ok] > 0)  # visibility is a decision
    # a flagged ceiling moves the radius by at most one pixel
    both = ~okv & (rg > 0) & (pr["radius"] > 0)
    assert (np.abs(rg[both] - pr["radius"][both]) <= 1).all()
    vis = ok & (pr["radius"] > 0)
    assert vis.sum() > 0
    # continuous outputs.  The camera-space coordinates come from fp32 sums R mu + t whose
    # terms can cancel (a mean far to the side, barely in front of the near plane), so the
    # bound on u, v, z scales with each sum's condition number sum|terms| / |result|.
    R = cam.R.astype(np.float64)
    mu = P[0, :, :3].astype(np.float64)
    terms = np.abs(mu @ R.T) + np.abs(cam.t.astype(np.float64))
    pc = mu @ R.T + cam.t.astype(np.float64)
    cond = terms / np.maximum(np.abs(pc), 1e-12)
    # u = fx x/z + cx: the two terms can cancel too (u near 0), so the bound is absolute,
    # built from the magnitude of each term
    for name, col, c0, ci in [("u", 0, cam.cx, 0), ("v", 1, cam.cy, 1)]:
        ref = pr["uvzo"][vis, col]
        term = np.abs(ref - c0)
        tol = 1e-6 * (term * (1.0 + cond[vis, ci] + cond[vis, 2]) + abs(c0))
        assert (np.abs(g[0, vis, col] - ref) <= tol).all(), name
    for name, a, b, rel in [("z", g[0, vis, 2], pr["uvzo"][vis, 2], 1e-6 * (1.0 + cond[vis, 2])),
                            ("o", g[0, vis, 3], pr["uvzo"][vis, 3], 1e-6)]:
        err = np.abs(a - b) / np.maximum(np.abs(b), 1.0)
        assert (err <= rel).all(), (name, err.max())
    # conic: error relative to the largest entry of the same Gaussian
    scale = np.abs(pr["conic"][vis]).max(axis=1, keepdims=True)
    cerr = np.abs(g[1, vis, :3] - pr["conic"][vis]) / scale
    assert cerr.max() <= 1e-4, cerr.max()
    assert np.abs(g[2, vis, :3] - pr["rgb"][vis]).max() <= 1e-5
    # culled Gaussians write zeros
    culled = ok & (pr["radius"] == 0)
    assert (g[:, culled] == 0).all()


def test_project_empty_and_single():
    P, cam = scene(0, 1)
    g = gpu_project(P, cam)
    pr = oracle.project(P, cam)
    assert g[1, 0, 3].view(np.int32) == pr["radius"][0]
    proj = torch.zeros((3, 1, 4), dtype=torch.float32, device="cuda")
    N.gs_project(dev(P), 0, cam, proj)  # n = 0 is a no-op
    with pytest.raises(N.GSError):
        N.gs_project(dev(P), -1, cam, proj)


@pytest.mark.parametrize("case", ["60k-mixed-sizes", "2k-18-views"])
def test_project_batch_matches_per_view(case):
    """gs_project_batch equals gs_project view by view, bit for bit (18 views: two launches)."""
    if case == "60k-mixed-sizes":
        P = scenes.make_params(1, n=60_000)
        cams = [scenes.make_cameras(1)[v] for v in (0, 17, 33)] + [scenes.make_cameras(3)[1]]
    else:
        P = scenes.make_params(1, n=2048)
        cams = scenes.make_cameras(1)[:18]
    n = P.shape[1]
    projs = [torch.full((3, n, 4), 7.0, dtype=torch.float32, device="cuda") for _ in cams]
    stride = (n + 31) // 32 + 3  # a padded row: the padding is never written
    bits = torch.full((len(cams), stride), -1, dtype=torch.int32, device="cuda")
    N.gs_project_batch(dev(P), n, cams, projs, visible_bits=bits, bits_stride=stride)
    torch.cuda.synchronize()
    hb = host(bits).view(np.uint32)
    for b, cam in enumerate(cams):
        single = gpu_project(P, cam)
        assert np.array_equal(host(projs[b]).view(np.uint32), single.view(np.uint32)), b
        # the visibility bitset: bit i of the view set iff its radius is > 0, bits past n clear
        vis = np.zeros(stride * 32 - 96, bool)
        vis[:n] = single[1, :, 3].view(np.int32) > 0
        want = np.packbits(vis.reshape(-1, 32)[:, ::-1], axis=1).view(">u4").ravel().astype(np.uint32)
        assert np.array_equal(hb[b, : stride - 3], want), b
        assert (hb[b, stride - 3:] == 0xFFFFFFFF).all()
    # and the first view against the oracle's integer decisions
    pr = oracle.project(P, cams[0])
    ok = (pr["margin"] >= MARGIN) & (pr["rmargin"] >= MARGIN)
    assert np.array_equal(host(projs[0])[1, ok, 3].view(np.int32), pr["radius"][ok])


# ------------------------------------------------------------------ binning + sort
@pytest.mark.parametrize("cfg,n,view", [(0, None, 0), (0, 1, 0), (0, 2047, 0), (0, 2049, 0), (1, 300_000, 5),
                                        (2, 200_000, 3), (3, 2_000_003, 0)])
def test_bin_sort_bit_exact(cfg, n, view):
    # (3, 2_000_003): from 2M Gaussians on, the depth passes use the wide radix tiles; about
    # 31 % of this view's Gaussians are culled and dropped by the first pass
    P, cam = scene(cfg, n, view)
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    keys_o, vals_o, ranges_o = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
    keys, vals, ranges, M, count = gpu_bin_sort(planes, cam)
    assert count[1] == 0
    assert M == len(keys_o)
    assert np.array_equal(keys, keys_o)
    assert np.array_equal(vals, vals_o)
    assert np.array_equal(ranges, ranges_o)
    if n is None or n > 100_000:  # without the keys output: same values and ranges, keys untouched
        keys2, vals2, ranges2, M2, count2 = gpu_bin_sort(planes, cam, with_keys=False)
        assert count2[1] == 0 and M2 == M and not keys2.any()
        assert np.array_equal(vals2, vals_o) and np.array_equal(ranges2, ranges_o)


def test_bin_sort_ties_keep_index_order():
    # every Gaussian at the same depth: order inside a tile must be by index
    P, cam = scene(0)
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    vis = planes[1, :, 3].view(np.int32) > 0
    planes[0, vis, 2] = 4.0
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    keys_o, vals_o, ranges_o = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
    keys, vals, ranges, M, _ = gpu_bin_sort(planes, cam)
    assert np.array_equal(keys, keys_o) and np.array_equal(vals, vals_o) and np.array_equal(ranges, ranges_o)


def test_bin_sort_all_culled_and_overflow():
    P, cam = scene(0)
    planes = np.zeros((3, P.shape[1], 4), np.float32)  # every radius 0
    keys, vals, ranges, M, count = gpu_bin_sort(planes, cam, capacity=16)
    assert M == 0 and count[1] == 0 and (ranges == 0).all()
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    with pytest.raises(N.GSError) as e:
        gpu_bin_sort(planes, cam, capacity=100)
    assert e.value.status == N.GS_ERR_CAPACITY


@pytest.mark.parametrize("mode", [1, 2], ids=["tile-sort-barrier", "depth-sort-barrier"])
def test_bin_sort_bounded_wait_reports_timeout(mode):
    """A flag that nothing sets (a grid-barrier arrival): every other CTA's wait gives up and
    reports, and the GPU stays usable."""
    P, cam = scene(1, 100_000, 0)
    planes = proj_planes_from_oracle(oracle.project(P, cam))
    N.gs_debug_set_wait_limit(2000)
    N.gs_debug_drop_publish(mode)
    try:
        with pytest.raises(N.GSError) as e:
            gpu_bin_sort(planes, cam)
        assert e.value.status == N.GS_ERR_TIMEOUT
    finally:
        N.gs_debug_drop_publish(0)
        N.gs_debug_set_wait_limit(0)
    keys, vals, ranges, M, count = gpu_bin_sort(planes, cam)  # next call is clean
    assert count[1] == 0 and M > 0


def gpu_bin_sort_batch(planes_list, cams, capacity=None, with_keys=True):
    n = planes_list[0].shape[1]
    B = len(cams)
    if capacity is None:
        capacity = max(int(p[2, :, 3].view(np.int32).astype(np.int64).sum()) for p in planes_list) + 1
    ws_bytes = N.gs_bin_sort_batch_workspace_size(B, n, capacity, cams)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    projs = [dev(p) for p in planes_list]
    keys = [torch.zeros(max(capacity, 1), dtype=torch.int64, device="cuda") for _ in range(B)]
    vals = [torch.zeros(max(capacity, 1), dtype=torch.int32, device="cuda") for _ in range(B)]
    ranges = [torch.full((c.tiles_x * c.tiles_y, 2), 7, dtype=torch.int32, device="cuda") for c in cams]
    counts = torch.zeros((B, 2), dtype=torch.int64, device="cuda")
    Ms = N.gs_bin_sort_batch(projs, n, cams, ws, ws_bytes, keys if with_keys else None, vals, capacity, ranges,
                             counts, sync=True)
    return [(host(keys[b])[:Ms[b]].view(np.uint64), host(vals[b])[:Ms[b]].view(np.uint32),
             host(ranges[b]).view(np.uint32), Ms[b]) for b in range(B)], host(counts)


def _batch_case(case):
    if case == "small-10-views":  # two launch groups: the second reuses the first's depth buffers
        P = scenes.make_params(1, n=2048)
        return P, scenes.make_cameras(1)[:10]
    if case == "300k-4-views":  # fewer CTAs per view than radix tiles of the depth sort
        P = scenes.make_params(1, n=300_000)
        return P, [scenes.make_cameras(1)[v] for v in (0, 5, 11, 23)]
    if case == "2m-2-views":  # wide depth radix tiles, views with different visible counts
        P = scenes.make_params(3, n=2_000_003)
        return P, [scenes.make_cameras(3)[v] for v in (0, 2)]
    # image sizes differ inside the batch (1236x820 and 1920x1080 cameras on one scene)
    P = scenes.make_params(1, n=50_000)
    return P, [scenes.make_cameras(1)[2], scenes.make_cameras(3)[0], scenes.make_cameras(1)[7]]


@pytest.mark.parametrize("case", ["small-10-views", "300k-4-views", "2m-2-views", "mixed-sizes"])
def test_bin_sort_batch_bit_exact(case):
    P, cams = _batch_case(case)
    planes_list = [proj_planes_from_oracle(oracle.project(P, c)) for c in cams]
    out, counts = gpu_bin_sort_batch(planes_list, cams)
    assert (counts[:, 1] == 0).all()
    for b, (planes, cam) in enumerate(zip(planes_list, cams)):
        uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
        keys_o, vals_o, ranges_o = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
        keys, vals, ranges, M = out[b]
        assert M == len(keys_o) == counts[b, 0], b
        assert np.array_equal(keys, keys_o), b
        assert np.array_equal(vals, vals_o), b
        assert np.array_equal(ranges, ranges_o), b


def test_bin_sort_batch_timeout_is_per_view():
    """View 0's depth-sort barrier never completes: view 0 reports the timeout, the other
    views of the launch finish cleanly and the next call is clean."""
    P = scenes.make_params(1, n=100_000)
    cams = [scenes.make_cameras(1)[v] for v in (0, 1, 2)]
    planes_list = [proj_planes_from_oracle(oracle.project(P, c)) for c in cams]
    N.gs_debug_set_wait_limit(2000)
    N.gs_debug_drop_publish(2)
    try:
        with pytest.raises(N.GSError) as e:
            gpu_bin_sort_batch(planes_list, cams)
        assert e.value.status == N.GS_ERR_TIMEOUT
    finally:
        N.gs_debug_drop_publish(0)
        N.gs_debug_set_wait_limit(0)
    out, counts = gpu_bin_sort_batch(planes_list, cams)
    assert (counts[:, 1] == 0).all() and all(o[3] > 0 for o in out)


# ------------------------------------------------------------------ compositing forward
def oracle_stage_chain(P, cam):
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    keys, vals, ranges = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
    return planes, (uvzo, conic, radius, rgb), keys, vals, ranges


def gpu_render(planes, vals, ranges, cam, bg=(0.0, 0.0, 0.0)):
    n = planes.shape[1]
    H, W = cam.height, cam.width
    img = torch.zeros((3, H, W), dtype=torch.float32, device="cuda")
    T = torch.zeros((H, W), dtype=torch.float32, device="cuda")
    nc = torch.zeros((H, W), dtype=torch.int32, device="cuda")
    v = vals if len(vals) else np.zeros(1, np.uint32)
    N.gs_render_fwd(dev(planes), n, dev(v.view(np.int32)), dev(ranges.view(np.int32)), cam, bg, img, T, nc)
    torch.cuda.synchronize()
    return host(img), host(T), host(nc).view(np.uint32)


@pytest.mark.parametrize("cfg,n,view,bg", [(0, None, 0, (0.0, 0.0, 0.0)), (0, None, 0, (0.2, 0.5, 1.0)),
                                           (1, 300_000, 2, (0.0, 0.0, 0.0))])
def test_render_fwd_parity(cfg, n, view, bg):
    P, cam = scene(cfg, n, view)
    planes, (uvzo, conic, radius, rgb), keys, vals, ranges = oracle_stage_chain(P, cam)
    img_o, T_o, nc_o, mg = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height, bg)
    img, T, nc = gpu_render(planes, vals, ranges, cam, bg)
    ok = mg >= MARGIN
    flagged = int((~ok).sum())
    report(f"render_fwd cfg{cfg} flagged pixels", flagged, ok.size)
    assert flagged <= max(2, FLAG_FRAC_PIXELS * ok.size)
    assert np.abs(img - img_o)[:, ok].max() <= IMG_ATOL
    # a flagged pixel differs by at most what one flipped decision can change
    if flagged:
        assert np.abs(img - img_o)[:, ~ok].max() <= flag_img_bound(rgb, bg)
    assert np.abs(T - T_o)[ok].max() <= IMG_ATOL
    assert np.array_equal(nc[ok], nc_o[ok])
    # compositing invariants on the CUDA output itself
    assert (T >= 1e-4 * (1 - 1e-6)).all() and (T <= 1.0).all()


def test_render_fwd_empty_tiles():
    P, cam = scene(0)
    planes = np.zeros((3, P.shape[1], 4), np.float32)
    ranges = np.zeros((cam.tiles_x * cam.tiles_y, 2), np.uint32)
    img, T, nc = gpu_render(planes, np.zeros(0, np.uint32), ranges, cam, (0.1, 0.2, 0.3))
    assert np.allclose(img[0], 0.1) and np.allclose(img[2], 0.3) and (T == 1).all() and (nc == 0).all()


def test_render_fwd_ragged_image():
    # width/height not multiples of 16: the last tile row/column is partial
    P = scenes.make_params(0)
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), 100, 71, 110.0)
    planes, (uvzo, conic, radius, rgb), keys, vals, ranges = oracle_stage_chain(P, cam)
    img_o, T_o, nc_o, mg = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height)
    img, T, nc = gpu_render(planes, vals, ranges, cam)
    ok = mg >= MARGIN
    assert np.abs(img - img_o)[:, ok].max() <= IMG_ATOL


# ------------------------------------------------------------------ loss
@pytest.mark.parametrize("H,W,scale", [(128, 128, 1.0), (37, 53, 0.25), (820, 1236, 0.25), (7, 5, 1.0),
                                     (1080, 1920, 0.25), (2160, 3840, 1.0 / 16)])
def test_loss_parity(H, W, scale):
    rng = np.random.default_rng(H * 1000 + W)
    x = rng.uniform(0, 1, size=(3, H, W)).astype(np.float32)
    y = np.clip(x + rng.normal(0, 0.1, size=x.shape), 0, 1).astype(np.float32)
    val_o, d_o = oracle.loss(x, y, scale=scale)
    ws_b = N.gs_loss_workspace_size(W, H)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    loss = torch.full((1,), 0.5, dtype=torch.float32, device="cuda")
    d = torch.zeros((3, H, W), dtype=torch.float32, device="cuda")
    N.gs_loss(dev(x), dev(y), W, H, 0.8, 0.2, scale, loss, False, d, ws, ws_b)
    torch.cuda.synchronize()
    assert float(loss.item()) == pytest.approx(val_o, rel=1e-5)
    dd = host(d)
    bad = allclose_grad(dd, d_o, RTOL, 1e-6 * np.abs(d_o).max())
    assert bad.sum() == 0, (np.abs(dd - d_o).max(), np.abs(d_o).max())
    # accumulate mode adds
    N.gs_loss(dev(x), dev(y), W, H, 0.8, 0.2, scale, loss, True, d, ws, ws_b)
    assert float(loss.item()) == pytest.approx(2 * val_o, rel=1e-5)


# ------------------------------------------------------------------ compositing backward
@pytest.mark.parametrize("ordered", [False, True], ids=["index-order", "heaviest-first"])
def test_render_bwd_parity_config0(ordered):
    P, cam = scene(0)
    planes, (uvzo, conic, radius, rgb), keys, vals, ranges = oracle_stage_chain(P, cam)
    img_o, T_o, nc_o, mg = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height)
    tgt = oracle.render_view(scenes.jitter_means(P, 0.02, 2000), cam)
    _, dimg = oracle.loss(img_o.astype(np.float32), tgt.astype(np.float32))
    # the image gradient is zeroed on both sides where a compositing decision sits on its
    # threshold: a decision flipped there then reaches no Gaussian, and nothing is set aside
    flagged = mg < MARGIN
    report("render_bwd cfg0 flagged pixels (gradient zeroed)", int(flagged.sum()), flagged.size)
    dimg32 = (dimg * ~flagged[None]).astype(np.float32)
    g_o = oracle.render_bwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height, dimg32.astype(np.float64))
    n = P.shape[1]
    grad2d = torch.full((n, 12), 3.0, dtype=torch.float32, device="cuda")  # the call clears it
    order = None
    if ordered:  # the trainer's backward launch order: by each tile's largest n_contrib
        Tn = cam.tiles_x * cam.tiles_y
        pad = np.zeros((cam.tiles_y * 16, cam.tiles_x * 16), np.int64)
        pad[:cam.height, :cam.width] = nc_o
        cost = pad.reshape(cam.tiles_y, 16, cam.tiles_x, 16).max(axis=(1, 3)).ravel().astype(np.int32)
        order = torch.zeros(Tn, dtype=torch.int32, device="cuda")
        N.gs_tile_order(None, dev(cost), cam.tiles_x, cam.tiles_y, order)
    N.gs_render_bwd(dev(planes), n, dev(vals.view(np.int32)), dev(ranges.view(np.int32)), cam, None,
                    dev(T_o.astype(np.float32)), dev(nc_o.view(np.int32)), dev(dimg32), grad2d, tile_order=order)
    torch.cuda.synchronize()
    g = host(grad2d)
    # columns: oracle (du, dv, dA, dB, dC, dop, dr, dg, db) vs gs (du, dv, dop, 0, dA, dB, dC, 0, dr, dg, db, 0)
    gm = grad2d_oracle_layout(g)
    assert (g[:, [3, 7, 11]] == 0).all()
    bad = allclose_grad(gm, g_o)
    report("render_bwd cfg0 (every Gaussian)", int(bad.sum()), bad.size)
    assert bad.sum() == 0


# ------------------------------------------------------------------ tile launch order
def cost_key(c):
    """gs_tile_order's documented ranking key: 0 for a zero cost, else 1 + 16 floor(log2 c)
    plus the four bits of c below its leading one."""
    c = np.asarray(c, np.int64)
    hb = np.where(c > 0, np.floor(np.log2(np.maximum(c, 1))).astype(np.int64), 0)
    frac = np.where(hb >= 4, (c >> np.maximum(hb - 4, 0)) & 15, (c << np.maximum(4 - hb, 0)) & 15)
    return np.where(c > 0, 1 + 16 * hb + frac, 0)


@pytest.mark.parametrize("tx,ty,block", [(1, 1, 4), (5, 3, 4), (77, 1, 4), (1, 77, 3), (78, 53, 4), (240, 135, 4),
                                         (240, 135, 1), (361, 361, 8), (100, 70, 2)])
def test_tile_order_is_a_heaviest_first_permutation(tx, ty, block):
    T = tx * ty
    rng = np.random.default_rng(T)
    cost = np.where(rng.random(T) < 0.2, 0, rng.integers(1, 1 << 20, T)).astype(np.int64)
    cost[:3] = [0, (1 << 31) + 5, 1][:min(3, T)]  # a zero, a cost past 2^31, a one
    starts = rng.integers(0, 1 << 30, T)
    ranges = np.stack([starts, starts + cost], 1).astype(np.uint32)
    ys, xs = np.divmod(np.arange(T), tx)
    ux = (tx + block - 1) // block
    blk = (ys // block) * ux + xs // block
    bkey = np.zeros(blk.max() + 1, np.int64)
    np.maximum.at(bkey, blk, cost_key(cost.astype(np.uint32).astype(np.int64)))
    for by_cost in (False, True):
        order = torch.full((T,), -1, dtype=torch.int32, device="cuda")
        N.gs_tile_order(None if by_cost else dev(ranges.view(np.int32)),
                        dev(cost.astype(np.uint32).view(np.int32)) if by_cost else None, tx, ty, order, block=block)
        torch.cuda.synchronize()
        o = host(order).view(np.uint32).astype(np.int64)
        assert np.array_equal(np.sort(o), np.arange(T))
        # square blocks of tiles, each contiguous and row-major inside, by falling key
        b = blk[o]
        starts_b = np.flatnonzero(np.r_[True, b[1:] != b[:-1]])
        assert len(starts_b) == len(bkey)  # every block appears as one run
        for s0, s1 in zip(starts_b, np.r_[starts_b[1:], T]):
            assert np.array_equal(o[s0:s1], np.sort(o[s0:s1]))
        assert (np.diff(bkey[b[starts_b]]) <= 0).all()
    N.gs_tile_order(None, None, 0, 5, None, block=block)  # nothing to order: no launch, no error


def test_render_with_tile_order_matches_index_order():
    """The launch order changes no forward result and the backward only by the order of its
    atomic sums; tile_cost is the largest n_contrib of each tile."""
    P, cam = scene(1, 300_000, 2)
    planes, (uvzo, conic, radius, rgb), keys, vals, ranges = oracle_stage_chain(P, cam)
    img0, T0, nc0 = gpu_render(planes, vals, ranges, cam)
    n, H, W = P.shape[1], cam.height, cam.width
    Tn = cam.tiles_x * cam.tiles_y
    dv, dr, dp = dev(vals.view(np.int32)), dev(ranges.view(np.int32)), dev(planes)
    order = torch.zeros((2, Tn), dtype=torch.int32, device="cuda")
    tcost = torch.full((Tn,), 7, dtype=torch.int32, device="cuda")
    img = torch.zeros((3, H, W), dtype=torch.float32, device="cuda")
    Tf = torch.zeros((H, W), dtype=torch.float32, device="cuda")
    nc = torch.zeros((H, W), dtype=torch.int32, device="cuda")
    N.gs_tile_order(dr, None, cam.tiles_x, cam.tiles_y, order[0])
    N.gs_render_fwd(dp, n, dv, dr, cam, None, img, Tf, nc, tile_order=order[0], tile_cost=tcost)
    torch.cuda.synchronize()
    assert np.array_equal(host(img), img0) and np.array_equal(host(Tf), T0)
    assert np.array_equal(host(nc).view(np.uint32), nc0)
    pad = np.zeros((cam.tiles_y * 16, cam.tiles_x * 16), np.int64)
    pad[:H, :W] = nc0
    assert np.array_equal(host(tcost).astype(np.int64), pad.reshape(cam.tiles_y, 16, cam.tiles_x, 16).max(axis=(1, 3)).ravel())
    N.gs_tile_order(None, tcost, cam.tiles_x, cam.tiles_y, order[1])
    rng = np.random.default_rng(5)
    dimg = dev(rng.normal(0, 1e-3, (3, H, W)).astype(np.float32))
    g = [torch.zeros((n, 12), dtype=torch.float32, device="cuda") for _ in range(2)]
    N.gs_render_bwd(dp, n, dv, dr, cam, None, Tf, nc, dimg, g[0])
    N.gs_render_bwd(dp, n, dv, dr, cam, None, Tf, nc, dimg, g[1], tile_order=order[1])
    torch.cuda.synchronize()
    a, b = host(g[0]), host(g[1])
    # the same fp32 terms summed in another order: a zero-mean image gradient makes many sums
    # cancel, so the bound is relative to each column's largest magnitude
    scale = np.abs(a).max(axis=0, keepdims=True)
    assert (np.abs(a - b) <= 1e-5 * scale + 1e-12).all()
    assert scale.max() > 0


# ------------------------------------------------------------------ projection backward
@pytest.mark.parametrize("cfg,n,view", [(0, None, 0), (1, 40_000, 9)])
def test_project_bwd_parity(cfg, n, view):
    P, cam = scene(cfg, n, view)
    pr = oracle.project(P, cam)
    planes = proj_planes_from_oracle(pr)
    n = P.shape[1]
    rng = np.random.default_rng(5)
    g2d = rng.normal(0, 1e-3, size=(n, 9)) * (pr["radius"] > 0)[:, None]
    g2d = g2d.astype(np.float32).astype(np.float64)
    ok = pr["margin"] >= MARGIN
    # the colour clamp at 0 switches the gradient off: keep away from raw colour ~ 0
    ok &= (np.abs(pr["raw"]) > 1e-4).all(axis=1) | (pr["radius"] == 0)
    g2d[~ok] = 0
    ref = oracle.project_bwd(P, cam, g2d)
    gs_layout = np.zeros((n, 12), np.float32)
    gs_layout[:, [0, 1, 4, 5, 6, 2, 8, 9, 10]] = g2d
    grads = torch.full((15, n, 4), 0.25, dtype=torch.float32, device="cuda")  # accumulates (+=)
    N.gs_project_bwd(dev(P), n, cam, dev(planes), dev(gs_layout), grads)
    torch.cuda.synchronize()
    g = host(grads).astype(np.float64) - 0.25
    bad = allclose_grad(g, ref, RTOL, 1e-6)
    bad[1, :, 3] = False  # padding lane
    report(f"project_bwd cfg{cfg}", int(bad.sum()), bad.size)
    assert bad.sum() == 0


# ------------------------------------------------------------------ Adam
def test_sparse_adam_parity_and_skip():
    rng = np.random.default_rng(9)
    n = 10_000
    P = rng.normal(size=(15, n, 4)).astype(np.float32)
    G = rng.normal(0, 1e-2, size=(15, n, 4)).astype(np.float32)
    M = rng.normal(0, 1e-3, size=(15, n, 4)).astype(np.float32)
    V = np.abs(rng.normal(0, 1e-4, size=(15, n, 4))).astype(np.float32)
    idx = np.sort(rng.choice(n, 3_000, replace=False)).astype(np.uint32)
    ref = oracle.sparse_adam(P, G, M, V, idx, 1e-3, 0.9, 0.999, 1e-15, 4, 7)
    tp, tg, tm, tv = dev(P), dev(G), dev(M), dev(V)
    nidx = torch.tensor([len(idx)], dtype=torch.int64, device="cuda")
    counts = torch.zeros((4, 2), dtype=torch.int64, device="cuda")
    N.gs_sparse_adam(tp, tg, tm, tv, n, dev(idx.view(np.int32)), nidx, n, 1e-3, 0.9, 0.999, 1e-15, 4, 7, counts, 4)
    torch.cuda.synchronize()
    for got, want in zip((tp, tg, tm, tv), ref):
        bad = allclose_grad(host(got), want, RTOL, ATOL)
        assert bad.sum() == 0
    # the update itself (p_new - p_old): relative 1e-3, plus the fp32 rounding of p_new
    pn = host(tp).astype(np.float64)
    d_gpu, d_ref = pn - P, ref[0] - P
    tol = RTOL * np.abs(d_ref) + 2.0 ** -22 * np.maximum(np.abs(P), np.abs(pn))
    assert (np.abs(d_gpu - d_ref) <= tol).all()
    untouched = np.setdiff1d(np.arange(n), idx)
    assert (host(tp)[:, untouched] == P[:, untouched]).all()
    assert (host(tg)[:, untouched] == G[:, untouched]).all()
    # a view with a nonzero status word: the whole update is skipped
    counts[2, 1] = 1
    before = host(tp).copy()
    N.gs_sparse_adam(tp, tg, tm, tv, n, dev(idx.view(np.int32)), nidx, n, 1e-3, 0.9, 0.999, 1e-15, 4, 8, counts, 4)
    torch.cuda.synchronize()
    assert (host(tp) == before).all()


# ------------------------------------------------------------------ batched backward + Adam
def test_project_bwd_adam_parity_and_skip():
    """gs_project_bwd_adam == sum over views of the oracle's projection backward, then the
    oracle's sparse Adam over the union of the visible sets."""
    P, cam0 = scene(1, 40_000, 0)
    P[0, :50, :3] = [0.0, 1e5, 0.0]  # far outside every view: must stay untouched
    n = P.shape[1]
    cams = [scenes.make_cameras(1)[v] for v in (0, 9, 17, 30)]
    rng = np.random.default_rng(21)
    planes, g2ds, G = [], [], np.zeros((15, n, 4))
    ok = np.ones(n, bool)
    vis_any = np.zeros(n, bool)
    for cam in cams:
        pr = oracle.project(P, cam)
        vis = pr["radius"] > 0
        ok &= pr["margin"] >= MARGIN
        ok &= (np.abs(pr["raw"]) > 1e-4).all(axis=1) | ~vis
        vis_any |= vis
        g2d = (rng.normal(0, 1e-3, size=(n, 9)) * vis[:, None]).astype(np.float32).astype(np.float64)
        planes.append(proj_planes_from_oracle(pr))
        g2ds.append(g2d)
    for cam, g2d in zip(cams, g2ds):
        g2d[~ok] = 0  # Gaussians near a discrete decision in some view carry no gradient
        G += oracle.project_bwd(P, cam, g2d)
    union = np.nonzero(vis_any)[0].astype(np.uint32)
    M = rng.normal(0, 1e-4, size=(15, n, 4)).astype(np.float32)
    V = np.abs(rng.normal(0, 1e-6, size=(15, n, 4))).astype(np.float32)
    ref_p, _, ref_m, ref_v = oracle.sparse_adam(P, G, M, V, union, 1e-3, 0.9, 0.999, 1e-15, len(cams), 5)
    tp, tm, tv = dev(P), dev(M), dev(V)
    dplanes = [dev(q) for q in planes]
    dg = []
    for g2d in g2ds:
        lay = np.zeros((n, 12), np.float32)
        lay[:, [0, 1, 4, 5, 6, 2, 8, 9, 10]] = g2d
        dg.append(dev(lay))
    counts = torch.zeros((len(cams), 2), dtype=torch.int64, device="cuda")
    N.gs_project_bwd_adam(tp, n, cams, dplanes, dg, tm, tv, 1e-3, 0.9, 0.999, 1e-15, 5, counts, len(cams))
    torch.cuda.synchronize()
    cmp = ok & vis_any
    # the gradient floor of the projection backward (ATOL) enters m scaled by 1 - beta1^B and
    # v by (1 - beta2^B) * 2|g|
    b1B, b2B = 1 - 0.9 ** len(cams), 1 - 0.999 ** len(cams)
    for name, got, want, floor in (("m", tm, ref_m, b1B * ATOL), ("v", tv, ref_v, b2B * 2 * np.abs(G) * ATOL + 1e-12)):
        floor = floor if np.isscalar(floor) else floor[:, cmp]
        bad = allclose_grad(host(got)[:, cmp], want[:, cmp], RTOL, floor)
        report(f"project_bwd_adam {name}", int(bad.sum()), bad.size)
        assert bad.sum() == 0
    pn = host(tp).astype(np.float64)
    d_gpu, d_ref = (pn - P)[:, cmp], (ref_p - P)[:, cmp]
    tol = RTOL * np.abs(d_ref) + 2.0 ** -22 * np.maximum(np.abs(P[:, cmp]), np.abs(pn[:, cmp])) + 1e-9
    bad = np.abs(d_gpu - d_ref) > tol
    report("project_bwd_adam params", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    # visible in no view: parameters and moments bit-for-bit untouched
    none = ~vis_any
    assert none.any()
    assert (host(tp)[:, none] == P[:, none]).all() and (host(tm)[:, none] == M[:, none]).all()
    assert (host(tv)[:, none] == V[:, none]).all()
    # a view with a nonzero status word: the whole update is skipped
    counts[3, 1] = 1
    before = [host(t).copy() for t in (tp, tm, tv)]
    N.gs_project_bwd_adam(tp, n, cams, dplanes, dg, tm, tv, 1e-3, 0.9, 0.999, 1e-15, 6, counts, len(cams))
    torch.cuda.synchronize()
    for t, b in zip((tp, tm, tv), before):
        assert (host(t) == b).all()
    # the visible sets' bitsets (left at the start of gs_visible_sets' workspace) in place of
    # the radius words: bit-identical results
    B = len(cams)
    ws = torch.empty(N.gs_visible_sets_workspace_size(B, n), dtype=torch.uint8, device="cuda")
    offs = torch.zeros(B + 1, dtype=torch.int64, device="cuda")
    idx = torch.zeros(B * n, dtype=torch.int32, device="cuda")
    uni = torch.zeros(n, dtype=torch.int32, device="cuda")
    nu = torch.zeros(1, dtype=torch.int64, device="cuda")
    inter = torch.zeros((B, B), dtype=torch.int64, device="cuda")
    jac = torch.zeros((B, B), dtype=torch.float32, device="cuda")
    N.gs_visible_sets(dplanes, B, n, ws, ws.numel(), offs, idx, uni, nu, inter, jac)
    counts[3, 1] = 0
    outs = []
    for bits in (None, ws):
        p2, m2, v2 = dev(P), dev(M), dev(V)
        N.gs_project_bwd_adam(p2, n, cams, dplanes, dg, m2, v2, 1e-3, 0.9, 0.999, 1e-15, 5, counts, B,
                              visible_bits=bits, bits_stride=(n + 31) // 32)
        torch.cuda.synchronize()
        outs.append([host(t) for t in (p2, m2, v2)])
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    with pytest.raises(N.GSError):
        N.gs_project_bwd_adam(tp, n, cams, dplanes, dg, tm, tv, 1e-3, 0.9, 0.999, 1e-15, 5, counts, B,
                              visible_bits=ws, bits_stride=(n + 31) // 32 - 1)


# ------------------------------------------------------------------ visible sets
@pytest.mark.parametrize("B,n", [(1, 1000), (4, 70_001), (16, 100_000)])
def test_visible_sets_bit_exact(B, n):
    rng = np.random.default_rng(B * 7 + n)
    radii = np.where(rng.uniform(size=(B, n)) < rng.uniform(0.05, 0.9, size=(B, 1)), rng.integers(1, 50, (B, n)), 0)
    if B > 1:
        radii[1] = 0  # an empty view
    radii = radii.astype(np.int32)
    projs = []
    for b in range(B):
        q = np.zeros((3, n, 4), np.float32)
        q[1, :, 3] = radii[b].view(np.float32)
        projs.append(dev(q))
    ws_b = N.gs_visible_sets_workspace_size(B, n)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    off = torch.zeros(B + 1, dtype=torch.int64, device="cuda")
    ind = torch.zeros(B * n, dtype=torch.int32, device="cuda")
    uni = torch.zeros(n, dtype=torch.int32, device="cuda")
    nu = torch.zeros(1, dtype=torch.int64, device="cuda")
    inter = torch.zeros((B, B), dtype=torch.int64, device="cuda")
    jac = torch.zeros((B, B), dtype=torch.float32, device="cuda")
    o_off, o_ind, o_uni, o_inter, o_jac = oracle.visible_sets(radii)
    # from the radius words, then from the same sets given as bitsets (no proj pointers)
    stride = (n + 31) // 32 + 1
    vis = np.zeros((B, stride * 32), bool)
    vis[:, :n] = radii > 0
    packed = np.packbits(vis.reshape(B, -1, 32)[:, :, ::-1], axis=2).view(">u4").reshape(B, stride)
    bits = dev(packed.astype(np.uint32).view(np.int32))
    for mode in ("radius", "bits"):
        for t in (off, ind, uni, nu, inter, jac):
            t.zero_()
        if mode == "radius":
            N.gs_visible_sets(projs, B, n, ws, ws_b, off, ind, uni, nu, inter, jac)
        else:
            N.gs_visible_sets(None, B, n, ws, ws_b, off, ind, uni, nu, inter, jac, visible_bits=bits,
                              bits_stride=stride)
        torch.cuda.synchronize()
        assert np.array_equal(host(off), o_off), mode
        assert np.array_equal(host(ind)[: o_off[-1]].view(np.uint32), o_ind), mode
        assert int(nu.item()) == len(o_uni), mode
        assert np.array_equal(host(uni)[: len(o_uni)].view(np.uint32), o_uni), mode
        assert np.array_equal(host(inter), o_inter), mode
        assert np.array_equal(host(jac), o_jac), mode


# ------------------------------------------------------------------ the whole step
def test_full_step_parity_config0():
    P, cam = scene(0)
    cfg = scenes.CONFIGS[0]
    tgt = oracle.render_view(scenes.jitter_means(P, cfg.jitter, 2000), cam).astype(np.float32)
    ref = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt[None], lr=cfg.lr, eps=cfg.eps)
    tr = Trainer(dev(P), cam.width, cam.height, 1, lr=cfg.lr, eps=cfg.eps)
    grads_before = None
    # gradients: run once without the update
    res = tr.step_async([cam], dev(tgt[None]), adam=False)
    torch.cuda.synchronize()
    assert (host(res.status)[:, 1] == 0).all()
    assert float(res.loss.item()) == pytest.approx(ref["loss"], rel=1e-5)
    grads_before = host(tr.grads).astype(np.float64)
    G = ref["grads"]
    # set aside only Gaussians whose own projection decision (cull, radius ceiling, tile
    # rectangle) sits within the margin of its threshold; every other entry must agree
    pr = oracle.project(P, cam)
    ok = pr["margin"] >= MARGIN
    report("step cfg0: Gaussians set aside", int((~ok).sum()), ok.size)
    assert (~ok).sum() <= max(2, FLAG_FRAC_GAUSSIANS * ok.size)
    bad = allclose_grad(grads_before, G)[:, ok]
    bad[1, :, 3] = False  # padding lane
    report("step grads cfg0", int(bad.sum()), bad.size)
    assert bad.sum() == 0
    # the update: at t = 1 each entry moves by lr' sign(g) (reading h3), so entries whose
    # oracle gradient lies within the 1e-6 floor of zero are not compared
    tr.grads.zero_()
    loss = tr.step([cam], dev(tgt[None]))
    assert loss == pytest.approx(ref["loss"], rel=1e-5)
    Pn = host(tr.params).astype(np.float64)
    clear = (np.abs(G) > 1e-6) & ok[None, :, None]
    bad = allclose_grad(Pn - P, ref["params"] - P, RTOL, 1e-6)[clear]
    report("step params cfg0", int(bad.sum()), bad.size)
    assert bad.sum() == 0


def test_step_with_host_targets_matches_device_targets():
    """Host targets are uploaded on a side stream, each view's loss waiting for its own copy:
    the loss is bit-identical to a step given device targets, and the update agrees up to
    the order of the backward's float atomics."""
    P = scenes.make_params(1, n=30_000)
    cams = [scenes.make_cameras(1)[v] for v in (2, 11, 23, 40)]
    rng = np.random.default_rng(4)
    tgt = rng.uniform(0, 1, size=(4, 3, cams[0].height, cams[0].width)).astype(np.float32)
    results = []
    for on_host in (False, True):
        tr = Trainer(dev(P), cams[0].width, cams[0].height, 4)
        t = torch.from_numpy(tgt).pin_memory() if on_host else dev(tgt)
        loss = tr.step(cams, t)
        torch.cuda.synchronize()
        results.append((loss, host(tr.params).astype(np.float64)))
    assert results[0][0] == results[1][0]
    # the gradient of the same batch: entries within the 1e-6 floor of zero can change sign
    # with the order of the backward's atomics, and at t = 1 Adam moves them by lr' sign(g)
    tr = Trainer(dev(P), cams[0].width, cams[0].height, 4)
    tr.step_async(cams, dev(tgt), adam=False)
    torch.cuda.synchronize()
    g = host(tr.grads)
    d0, d1 = results[0][1] - P, results[1][1] - P
    clear = np.abs(g) > 1e-6
    bad = (np.abs(d1 - d0) > RTOL * np.abs(d0) + 1e-7) & clear
    report("host-target step params", int(bad.sum()), int(clear.sum()))
    assert bad.sum() == 0
