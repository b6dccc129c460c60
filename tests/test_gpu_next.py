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
