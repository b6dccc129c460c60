"""Parity of the scheduling helpers with the CPU oracle (GB300 only): the balanced tile split
of the Grendel-GS notes (§3.1) and the greedy view order by the Odin summary's scheduling score.

Integer outputs (tile costs, cumulative sums, split points, view order) are compared bit for
bit; the scores are float32 sums taken in the same order on both sides, so they match
exactly too.  Every input comes from the scene generator or the oracle, never the CUDA path.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

import oracle  # noqa: E402
import scenes  # noqa: E402
from gaussian_splatting_gb300 import _native as N  # noqa: E402

from parity import oracle_inputs_from_planes, proj_planes_from_oracle  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    N.load()


def gpu_tile_split(cost, parts):
    H, W = cost.shape
    T = ((W + 15) // 16) * ((H + 15) // 16)
    c = torch.from_numpy(np.ascontiguousarray(cost, np.uint32).view(np.int32)).cuda()
    tc = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    cum = torch.full((T,), -1, dtype=torch.int64, device="cuda")
    bounds = torch.full((parts + 1,), -1, dtype=torch.int64, device="cuda")
    N.gs_tile_split(c, W, H, parts, tc, cum, bounds)
    torch.cuda.synchronize()
    return (tc.cpu().numpy().view(np.uint64), cum.cpu().numpy().view(np.uint64), bounds.cpu().numpy())


@pytest.mark.parametrize("H,W,K,seed", [(820, 1236, 8, 0), (128, 128, 3, 1), (2160, 3840, 64, 2), (17, 33, 1, 3),
                                        (822, 1237, 1024, 4)])
def test_tile_split_random_costs(H, W, K, seed):
    rng = np.random.default_rng(seed)
    cost = rng.integers(0, 10_000, size=(H, W), dtype=np.uint32)
    cost[rng.random((H, W)) < 0.3] = 0
    got = gpu_tile_split(cost, K)
    want = oracle.tile_split(cost, K)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


def test_tile_split_degenerate_costs():
    for cost in (np.zeros((64, 80), np.uint32), np.full((64, 96), 3, np.uint32)):
        got = gpu_tile_split(cost, 4)
        want = oracle.tile_split(cost, 4)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)


def test_tile_split_on_a_rendered_cost_map():
    # the per-pixel list length of an oracle render: a real sky / dense-region profile
    P = scenes.make_params(1, n=20_000)
    cam = scenes.make_cameras(1)[3]
    planes = proj_planes_from_oracle(oracle.project(P, cam))
    uvzo, conic, radius, rgb = oracle_inputs_from_planes(planes)
    keys, vals, ranges = oracle.bin_sort(uvzo, radius, cam.width, cam.height)
    _, _, n_contrib, _ = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cam.width, cam.height)
    cost = n_contrib.astype(np.uint32)
    assert cost.any()
    for K in (2, 8, 64):
        got = gpu_tile_split(cost, K)
        want = oracle.tile_split(cost, K)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)


def gpu_view_order(w, unit):
    B = w.shape[0]
    wd = torch.from_numpy(np.ascontiguousarray(w, np.float32)).cuda()
    order = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    score = torch.full((B,), -1.0, dtype=torch.float32, device="cuda")
    N.gs_view_order(wd, B, unit, order, score)
    torch.cuda.synchronize()
    return order.cpu().numpy(), score.cpu().numpy()


@pytest.mark.parametrize("unit", [1, 2, 3])
def test_view_order_on_jaccard_of_real_views(unit):
    # the Jaccard weights of sixteen views of a city fly-through (graded overlaps), from the
    # oracle's visible sets
    P = scenes.make_params(3, n=20_000)
    cams = scenes.make_cameras(3)[:16]
    radii = np.stack([oracle.project(P, c)["radius"] for c in cams])
    _, _, _, _, jac = oracle.visible_sets(radii)
    o_g, s_g = gpu_view_order(jac, unit)
    o_w, s_w = oracle.view_order(jac, unit)
    assert np.array_equal(o_g, o_w)
    assert np.array_equal(s_g.view(np.uint32), s_w.view(np.uint32))


@pytest.mark.parametrize("B,unit,seed", [(64, 1, 0), (64, 8, 1), (33, 5, 2), (1, 1, 3), (16, 16, 4)])
def test_view_order_random_weights(B, unit, seed):
    rng = np.random.default_rng(seed)
    w = rng.random((B, B)).astype(np.float32)
    w = np.round((w + w.T) / 2, 2).astype(np.float32)  # symmetric, with ties
    np.fill_diagonal(w, 1.0)
    o_g, s_g = gpu_view_order(w, unit)
    o_w, s_w = oracle.view_order(w, unit)
    assert np.array_equal(o_g, o_w)
    assert np.array_equal(s_g.view(np.uint32), s_w.view(np.uint32))


# ------------------------------------------------------------------ opacity pruning
def _random_sets(n, seed):
    rng = np.random.default_rng(seed)
    sets = [rng.standard_normal((15, n, 4)).astype(np.float32) for _ in range(3)]
    if n > 7:
        sets[0][0, 3, 3] = np.nan          # dropped
        sets[0][0, 7, 3] = np.float32(-0.5)  # exactly on the threshold below: kept
    return sets


def gpu_prune(sets, min_logit):
    n = sets[0].shape[1]
    ins = [torch.from_numpy(s).cuda() for s in sets]
    ws = torch.empty(max(N.gs_prune_workspace_size(n), 256), dtype=torch.uint8, device="cuda")
    nk = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    k = N.gs_prune(ins, n, min_logit, None, 0, ws, nk, sync=True)
    outs = [torch.full((15, max(k, 1), 4), 7.0, dtype=torch.float32, device="cuda") for _ in sets]
    if k > 0:
        assert N.gs_prune(ins, n, min_logit, outs, k, ws, nk, sync=True) == k
    return k, [o.cpu().numpy()[:, :k] for o in outs]


@pytest.mark.parametrize("n,seed", [(1, 0), (255, 1), (256, 2), (257, 3), (100_000, 4), (1_000_003, 5)])
def test_prune_matches_oracle(n, seed):
    sets = _random_sets(n, seed)
    t = float(np.float32(-0.5))
    k, got = gpu_prune(sets, t)
    kw, want = oracle.prune(sets, t)
    assert k == kw
    for g, w in zip(got, want):
        assert np.array_equal(g.view(np.uint32), w.view(np.uint32))


def test_prune_capacity_and_empty():
    sets = _random_sets(1000, 6)
    n = 1000
    ins = [torch.from_numpy(s).cuda() for s in sets]
    ws = torch.empty(max(N.gs_prune_workspace_size(n), 256), dtype=torch.uint8, device="cuda")
    nk = torch.zeros(1, dtype=torch.int64, device="cuda")
    outs = [torch.zeros((15, 10, 4), dtype=torch.float32, device="cuda") for _ in sets]
    with pytest.raises(N.GSError) as e:
        N.gs_prune(ins, n, -np.inf, outs, 10, ws, nk, sync=True)
    keep = ~np.isnan(sets[0][0, :, 3])  # everything but the NaN logit is >= -inf
    assert e.value.status == N.GS_ERR_CAPACITY and int(nk.item()) == int(keep.sum()) == 999
    assert np.array_equal(outs[0].cpu().numpy(), sets[0][:, keep][:, :10])  # the slots that fit
    empty = torch.zeros((15, 0, 4), dtype=torch.float32, device="cuda")
    assert N.gs_prune([empty], 0, 0.0, None, 0, None, nk, sync=True) == 0


def test_trainer_prune_then_step():
    from gaussian_splatting_gb300.trainer import Trainer
    P = scenes.make_params(1, n=20_000)
    P[0, ::3, 3] = -6.0  # a third of the Gaussians at opacity ~0.0025
    cams = scenes.make_cameras(1)[:2]
    tr = Trainer(torch.from_numpy(P).cuda(), cams[0].width, cams[0].height, 2)
    tr.exp_avg.normal_()
    tr.exp_avg_sq.uniform_()
    sets = [tr.params.cpu().numpy(), tr.exp_avg.cpu().numpy(), tr.exp_avg_sq.cpu().numpy()]
    k = tr.prune(0.005)
    kw, want = oracle.prune(sets, float(np.float32(np.log(0.005 / 0.995))))
    assert k == kw == tr.n and 0 < k < 20_000
    for g, w in zip((tr.params, tr.exp_avg, tr.exp_avg_sq), want):
        assert np.array_equal(g.cpu().numpy().view(np.uint32), w.view(np.uint32))
    targets = torch.rand((2, 3, cams[0].height, cams[0].width), device="cuda")
    loss = tr.step(cams, targets)  # the resized trainer runs a whole step
    assert np.isfinite(loss) and int(tr.counts[:, 1].abs().sum()) == 0


# ------------------------------------------------------------------ densification: clone / split
def _densify_inputs(n, seed):
    rng = np.random.default_rng(seed)
    P = rng.normal(size=(15, n, 4)).astype(np.float32)
    P[1, :, :3] = rng.uniform(-4.0, -1.0, size=(n, 3))
    P[1, :, 3] = 0.0
    M = rng.normal(size=(15, n, 4)).astype(np.float32)
    V = np.abs(rng.normal(size=(15, n, 4))).astype(np.float32)
    stat = np.zeros((n, 2), np.float32)
    stat[:, 1] = rng.integers(0, 5, size=n)
    stat[:, 0] = (rng.uniform(0, 2e-3, size=n) * stat[:, 1]).astype(np.float32)
    Z = rng.standard_normal((n, 6)).astype(np.float32)
    return P, M, V, stat, Z


def gpu_densify(P, M, V, stat, thr, lthr, Z):
    n = P.shape[1]
    d = [torch.from_numpy(a).cuda() for a in (P, M, V, stat, Z)]
    ws = torch.empty(max(N.gs_densify_workspace_size(n), 256), dtype=torch.uint8, device="cuda")
    counts = torch.full((3,), -1, dtype=torch.int64, device="cuda")
    total, nc, ns = N.gs_densify(d[0], d[1], d[2], n, d[3], thr, lthr, d[4], None, 0, ws, counts, sync=True)
    outs = [torch.full((15, max(total, 1), 4), 7.0, dtype=torch.float32, device="cuda") for _ in range(3)]
    if total:
        N.gs_densify(d[0], d[1], d[2], n, d[3], thr, lthr, d[4], outs, total, ws, counts, sync=True)
    return (total, nc, ns), [o.cpu().numpy()[:, :total] for o in outs]


@pytest.mark.parametrize("n,seed", [(1, 0), (255, 1), (257, 2), (100_000, 3), (1_000_003, 4)])
def test_densify_matches_oracle(n, seed):
    """Counts and layout bit-exact (kept Gaussians and clones are copies, new moments zero),
    split children within the parameter tolerance."""
    P, M, V, stat, Z = _densify_inputs(n, seed)
    thr, lthr = float(np.float32(8e-4)), float(np.float32(-2.5))
    (total, nc, ns), (gp, gm, gv) = gpu_densify(P, M, V, stat, thr, lthr, Z)
    (op, om, ov), (onc, ons) = oracle.densify(P, M, V, stat, thr, lthr, Z)
    assert (total, nc, ns) == (op.shape[1], onc, ons)
    if n >= 1000:
        assert nc > 0 and ns > 0
    kept = n - ns
    n_plain = kept + nc  # kept Gaussians, then the clones and split children in index order
    new_kind = []
    cnt = stat[:, 1]
    avg = np.where(cnt > 0, stat[:, 0] / np.where(cnt > 0, cnt, 1), 0).astype(np.float32)
    sel = np.nonzero((cnt > 0) & (avg >= np.float32(thr)))[0]
    for i in sel:
        new_kind += [1] if P[1, i, :3].max() <= np.float32(lthr) else [2, 2]
    exact = np.ones(total, bool)
    exact[kept:][np.array(new_kind, int) == 2] = False  # split children are recomputed in fp32
    assert np.array_equal(gp[:, exact].astype(np.float64), op[:, exact])
    assert np.array_equal(gm.astype(np.float64), om) and np.array_equal(gv.astype(np.float64), ov)
    if (~exact).any():
        bad = np.abs(gp[:, ~exact] - op[:, ~exact]) > 1e-6 * np.abs(op[:, ~exact]) + 1e-6
        assert bad.sum() == 0
    del n_plain


def test_densify_statistic_from_the_backward_passes():
    """gs_project_bwd and the fused gs_project_bwd_adam add |(dL/du, dL/dv)| and one view per
    visible Gaussian, as the oracle's statistic does on the same screen-space gradients."""
    P = scenes.make_params(1, n=50_000)
    cams = [scenes.make_cameras(1)[v] for v in (1, 9, 30)]
    n = P.shape[1]
    rng = np.random.default_rng(12)
    planes, g2ds, want = [], [], np.zeros((n, 2))
    ok = np.ones(n, bool)  # the kernels recompute the projection: skip decisions on a threshold
    for cam in cams:
        pr = oracle.project(P, cam)
        ok &= pr["margin"] >= 1e-5
        g2d = (rng.normal(0, 1e-3, size=(n, 9)) * (pr["radius"] > 0)[:, None]).astype(np.float32)
        planes.append(proj_planes_from_oracle(pr))
        g2ds.append(g2d)
        want = oracle.densify_stat(g2d.astype(np.float64), pr["radius"], want)
    lay = lambda g: np.ascontiguousarray(np.pad(g, ((0, 0), (0, 3)))[:, [0, 1, 5, 9, 2, 3, 4, 10, 6, 7, 8, 11]])
    dP = torch.from_numpy(P).cuda()
    stat = torch.zeros((n, 2), dtype=torch.float32, device="cuda")
    grads = torch.zeros((15, n, 4), dtype=torch.float32, device="cuda")
    for cam, pl, g in zip(cams, planes, g2ds):
        N.gs_project_bwd(dP, n, cam, torch.from_numpy(pl).cuda(), torch.from_numpy(lay(g)).cuda(), grads, stat)
    s_seq = stat.cpu().numpy()
    stat2 = torch.zeros((n, 2), dtype=torch.float32, device="cuda")
    m, v = torch.zeros_like(dP), torch.zeros_like(dP)
    N.gs_project_bwd_adam(dP.clone(), n, cams, [torch.from_numpy(pl).cuda() for pl in planes],
                          [torch.from_numpy(lay(g)).cuda() for g in g2ds], m, v, 1e-3, 0.9, 0.999, 1e-15, 1,
                          densify_stat=stat2)
    s_fused = stat2.cpu().numpy()
    torch.cuda.synchronize()
    for s in (s_seq, s_fused):
        assert np.array_equal(s[ok, 1], want[ok, 1])
        assert np.allclose(s[ok, 0], want[ok, 0], rtol=1e-6, atol=1e-12)
    assert (want[:, 1] == 3).sum() > 1000


def test_trainer_densify_then_step():
    from gaussian_splatting_gb300.trainer import Trainer
    P = scenes.make_params(1, n=30_000)
    cams = scenes.make_cameras(1)[:4]
    tr = Trainer(torch.from_numpy(P).cuda(), cams[0].width, cams[0].height, 4)
    targets = torch.rand((4, 3, cams[0].height, cams[0].width), device="cuda")
    for _ in range(2):
        tr.step(cams, targets)
    st = tr.dstat.cpu().numpy()
    assert (st[:, 1] == 8).sum() > 1000  # seen in all four views of both steps
    avg = st[:, 0] / np.maximum(st[:, 1], 1)
    thr = float(np.quantile(avg[st[:, 1] > 0], 0.9))  # about a tenth of the seen Gaussians
    params0 = tr.params.cpu().numpy()
    total, nc, ns = tr.densify(thr, 0.03, seed=5)
    assert nc > 0 and ns > 0 and total == 30_000 + nc + ns == tr.n
    assert tr.params.shape == (15, total, 4) and float(tr.dstat.abs().sum()) == 0.0
    kept = tr.params.cpu().numpy()[:, : total - nc - 2 * ns]
    assert np.isin(kept[0, :, 0], params0[0, :, 0]).all()
    loss = tr.step(cams, targets)  # the grown trainer runs a whole step
    assert np.isfinite(loss) and int(tr.counts[:, 1].abs().sum()) == 0
