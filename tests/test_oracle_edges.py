"""Pins of the oracle's edge behaviour: the 0.99 alpha cap, a non-zero background, equal
depth keys in the binning sort, Adam's epsilon, and the update set of a multi-view step.

Each case has a closed form written out here from the method's definition (one Gaussian
composited over a background; Adam's first step; a stable sort of instances generated in
index order; the union of the views' visible sets), so that a mistake in the oracle on one of
these paths fails a test even where the other pins never reach the path.
"""
import math

import numpy as np
import pytest

import oracle
import scenes

F32_ALPHA_CAP = float(np.float32(0.99))
F32_ALPHA_MIN = np.float32(1.0 / 255.0)


def _one_gaussian_pixels(W, H, ranges):
    """Pixels of the tiles whose list holds the one Gaussian (16x16 tiles, row-major)."""
    tx = (W + 15) // 16
    for t in np.nonzero(ranges[:, 1] > ranges[:, 0])[0]:
        x0, y0 = (int(t) % tx) * 16, (int(t) // tx) * 16
        for py in range(y0, min(y0 + 16, H)):
            for px in range(x0, min(x0 + 16, W)):
                yield px, py


# ------------------------------------------------------------------ alpha cap and background
def test_opaque_gaussian_over_background_closed_form():
    """One isotropic, nearly opaque Gaussian in front of a coloured background: every pixel is
    a * c + (1 - a) * bg with a = min(0.99, o G), pixels whose a is below 1/255 and pixels of
    tiles the Gaussian does not reach show the background, and the final transmittance is
    1 - a."""
    W = H = 128
    f = 140.0
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), W, H, f)
    P = np.zeros((15, 1, 4), np.float32)
    P[1, 0, :3] = -1.0
    P[0, 0, 3] = 6.0  # o = 0.9975: the centre is capped at 0.99
    P[2, 0, 0] = 1.0
    P[3, 0, :3] = (0.9, 0.2, 0.4)
    bg = (0.2, 0.5, 0.9)
    s = math.exp(np.float32(-1.0))
    o = 1.0 / (1.0 + math.exp(-6.0))
    var = (f * s / 4.0) ** 2 + 0.3
    colour = 0.5 / math.sqrt(math.pi) * np.array([float(np.float32(c)) for c in (0.9, 0.2, 0.4)]) + 0.5
    pr = oracle.project(P, cam)
    keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], W, H)
    img, T, nc, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, W, H, bg)
    expect = np.broadcast_to(np.asarray(bg)[:, None, None], (3, H, W)).copy()
    expect_T = np.ones((H, W))
    capped = 0
    for px, py in _one_gaussian_pixels(W, H, ranges):
        rho2 = (px + 0.5 - 64) ** 2 + (py + 0.5 - 64) ** 2
        oa = o * math.exp(-rho2 / (2 * var))
        a = F32_ALPHA_CAP if np.float32(oa) > np.float32(0.99) else oa
        capped += a == F32_ALPHA_CAP
        if np.float32(a) < F32_ALPHA_MIN:
            continue
        expect[:, py, px] = colour * a + (1 - a) * np.asarray(bg)
        expect_T[py, px] = 1 - a
    assert capped >= 4
    assert np.allclose(img, expect, atol=1e-12)
    assert np.allclose(T, expect_T, atol=1e-12)


def test_compositing_backward_one_gaussian_closed_form():
    """Reverse mode of C = a c + (1 - a) bg for one anisotropic Gaussian, pixel by pixel:
    dc = a dC; dL/da = (c - bg) . dC; where a = o G is below the cap, do += dL/da G and the
    exponent's gradient dL/da o G reaches the conic (-dx^2 / 2, -dx dy, -dy^2 / 2) and the
    screen position (A dx + B dy, B dx + C dy); where a is capped at 0.99 nothing but the
    colour has a gradient."""
    W, H = 48, 40
    u, v, o = 21.3, 17.8, 0.9995
    A, B, C = 0.006, -0.0025, 0.009
    rgb = np.array([[0.7, 0.3, 0.55]])
    bg = np.array([0.15, 0.6, 0.35])
    uvzo = np.array([[u, v, 2.0, o]])
    conic = np.array([[A, B, C]])
    radius = np.array([23], np.int32)
    keys, vals, ranges = oracle.bin_sort(uvzo, radius, W, H)
    dimg = np.random.default_rng(31).standard_normal((3, H, W))
    g2d = oracle.render_bwd(uvzo, conic, rgb, vals, ranges, W, H, dimg, bg)
    e = np.zeros(9)
    capped = 0
    for px, py in _one_gaussian_pixels(W, H, ranges):
        dx, dy = px + 0.5 - u, py + 0.5 - v
        power = -0.5 * (A * dx * dx + C * dy * dy) - B * dx * dy
        G = math.exp(power)
        cap = np.float32(o * G) > np.float32(0.99)
        a = F32_ALPHA_CAP if cap else o * G
        if np.float32(a) < F32_ALPHA_MIN:
            continue
        dC = dimg[:, py, px]
        e[6:9] += a * dC
        if cap:
            capped += 1
            continue
        da = float(np.dot(rgb[0] - bg, dC))
        e[5] += da * G
        dp = da * o * G
        e[2] += dp * (-0.5 * dx * dx)
        e[3] += dp * (-dx * dy)
        e[4] += dp * (-0.5 * dy * dy)
        e[0] += dp * (A * dx + B * dy)
        e[1] += dp * (B * dx + C * dy)
    assert capped >= 4
    assert np.allclose(g2d[0], e, rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("seed", [14])
def test_gradients_with_background_match_central_differences(seed):
    """Central differences of the whole step's loss with a coloured background (several
    Gaussians per pixel: the background enters every Gaussian's opacity gradient through the
    light that passes all of them)."""
    P, cam = scenes.tiny_scene(6, seed, width=32, height=32, focal=40.0)
    P = P.astype(np.float64)
    tgt = np.random.default_rng(seed + 100).uniform(0.0, 1.0, size=(1, 3, 32, 32))
    bg = (0.3, 0.8, 0.1)
    res = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt, bg=bg, do_adam=False)
    loss = lambda Q: oracle.step(Q, np.zeros_like(P), np.zeros_like(P), [cam], tgt, bg=bg, do_adam=False)["loss"]
    checked = 0
    for i in range(P.shape[1]):
        for plane, lane in ((0, 0), (0, 1), (0, 2), (0, 3), (1, 0), (2, 1), (3, 0), (3, 2)):
            h = 1e-5 * max(1.0, abs(P[plane, i, lane]))
            Pp, Pm = P.copy(), P.copy()
            Pp[plane, i, lane] += h
            Pm[plane, i, lane] -= h
            num = (loss(Pp) - loss(Pm)) / (2 * h)
            ana = res["grads"][plane, i, lane]
            assert abs(num - ana) <= 1e-4 * abs(num) + 1e-9, (i, plane, lane, num, ana)
            checked += 1
    assert checked == 48


# ------------------------------------------------------------------ binning: equal keys
def test_binning_equal_depths_keep_index_order():
    """Instances are generated in Gaussian index order and sorted stably by (tile, depth):
    among equal keys the Gaussian indices ascend, and each Gaussian appears once per tile of
    the square of half-width r around its (exactly representable) screen position."""
    rng = np.random.default_rng(41)
    W, H, N = 64, 48, 400
    u = rng.integers(0, W * 8, N) / 8.0
    v = rng.integers(0, H * 8, N) / 8.0
    z = rng.choice([1.0, 2.5, 4.0], N)  # three depths: long runs of equal keys
    r = rng.integers(1, 25, N).astype(np.int32)
    uvzo = np.stack([u, v, z, np.full(N, 0.5)], 1)
    keys, vals, ranges = oracle.bin_sort(uvzo, r, W, H)
    tx, ty = (W + 15) // 16, (H + 15) // 16
    expect = []
    for i in range(N):
        x0, x1 = max(0, math.floor((u[i] - r[i]) / 16)), min(tx, math.floor((u[i] + r[i]) / 16) + 1)
        y0, y1 = max(0, math.floor((v[i] - r[i]) / 16)), min(ty, math.floor((v[i] + r[i]) / 16) + 1)
        zb = int(np.float32(z[i]).view(np.uint32))
        for t_y in range(y0, y1):
            for t_x in range(x0, x1):
                expect.append((((t_y * tx + t_x) << 32) | zb, i))
    expect.sort(key=lambda e: e[0])  # stable
    assert keys.tolist() == [e[0] for e in expect]
    assert vals.tolist() == [e[1] for e in expect]
    runs = sum(1 for j in range(1, len(expect)) if expect[j][0] == expect[j - 1][0])
    assert runs > len(expect) // 2


# ------------------------------------------------------------------ Adam: epsilon
def test_adam_first_step_with_large_epsilon():
    """At t = 1 the bias-corrected moments are g and g^2, so the step is
    lr sqrt(b) g / (|g| + eps): epsilon is added after the square root."""
    rng = np.random.default_rng(43)
    N = 3
    P = rng.standard_normal((15, N, 4))
    G = rng.standard_normal((15, N, 4)) * np.array([0.01, 0.3, 1.0, 4.0])
    lr, b1, b2, eps, b = 0.05, 0.9, 0.999, 0.5, 4
    p, _, m, v = oracle.sparse_adam(P, G, np.zeros_like(P), np.zeros_like(P), list(range(N)), lr, b1, b2, eps, b, 1)
    assert np.allclose(p, P - lr * math.sqrt(b) * G / (np.abs(G) + eps), rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ the step's update set
def test_step_updates_the_union_of_the_views_visible_sets():
    """A two-view step updates exactly the Gaussians that either view sees: those seen only by
    the second view change too, those seen by neither keep their parameters and moments."""
    rng = np.random.default_rng(47)
    n = 24
    P = np.zeros((15, n, 4))
    P[0, :, 0] = np.linspace(-6.0, 6.0, n)
    P[0, :, 1] = rng.uniform(-0.3, 0.3, n)
    P[0, :, 2] = rng.uniform(-0.3, 0.3, n)
    P[0, :, 3] = rng.uniform(-1.0, 1.0, n)
    P[1, :, :3] = -2.0
    q = rng.standard_normal((n, 4))
    P[2] = q / np.linalg.norm(q, axis=1, keepdims=True)
    P[3, :, :3] = 0.4
    P = P.astype(np.float32).astype(np.float64)
    W = H = 32
    cams = [scenes.look_at((-4.0, 0.0, -3.0), (-4.0, 0.0, 0.0), W, H, 30.0),
            scenes.look_at((1.5, 0.0, -3.0), (1.5, 0.0, 0.0), W, H, 30.0)]
    seen = [oracle.project(P, c)["radius"] > 0 for c in cams]
    only_second = np.nonzero(seen[1] & ~seen[0])[0]
    neither = np.nonzero(~seen[0] & ~seen[1])[0]
    assert only_second.size and neither.size and seen[0].any()
    union = np.nonzero(seen[0] | seen[1])[0]
    tgt = rng.uniform(size=(2, 3, H, W))
    m0 = rng.uniform(0.0, 0.1, P.shape)
    v0 = rng.uniform(0.0, 0.1, P.shape)
    kw = dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, t=3)
    grads = oracle.step(P, m0, v0, cams, tgt, do_adam=False, **kw)["grads"]
    res = oracle.step(P, m0, v0, cams, tgt, do_adam=True, **kw)
    p, _, m, v = oracle.sparse_adam(P, grads, m0, v0, union.tolist(), 1e-2, 0.9, 0.999, 1e-8, 2, 3)
    assert np.array_equal(res["params"], p) and np.array_equal(res["m"], m) and np.array_equal(res["v"], v)
    assert (res["params"][:, only_second] != P[:, only_second]).any()
    assert np.array_equal(res["params"][:, neither], P[:, neither])
    assert np.array_equal(res["m"][:, neither], m0[:, neither])


# ------------------------------------------------------------------ clamped colour channel
def test_clamped_colour_channel_passes_no_gradient():
    """A colour channel whose SH sum + 0.5 is negative is clamped to 0, so near the parameters
    the loss does not depend on that channel's 16 coefficients (their gradient is exactly 0)
    and the view direction reaches the loss only through the other channels (the mean's
    gradient matches central differences)."""
    P, cam = scenes.tiny_scene(6, 14, width=32, height=32, focal=40.0)
    P = P.astype(np.float64)
    P[3, 0, 0] = -3.0  # sh[0][red]: 0.282 * -3 + 0.5 < 0
    for kk in range(1, 16):
        f = 3 * kk
        P[3 + f // 4, 0, f % 4] = 0.05 * ((-1) ** kk)
    pr = oracle.project(P, cam)
    assert pr["radius"][0] > 0 and pr["raw"][0, 0] < -0.2 and pr["rgb"][0, 0] == 0.0
    tgt = np.random.default_rng(114).uniform(0.0, 1.0, size=(1, 3, 32, 32))
    res = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)
    G = res["grads"]
    for kk in range(16):
        f = 3 * kk
        assert G[3 + f // 4, 0, f % 4] == 0.0, kk
    assert np.abs(G[3:, 0]).max() > 0  # the other channels do get gradients
    loss = lambda Q: oracle.step(Q, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)["loss"]
    for lane in range(3):
        h = 1e-5 * max(1.0, abs(P[0, 0, lane]))
        Pp, Pm = P.copy(), P.copy()
        Pp[0, 0, lane] += h
        Pm[0, 0, lane] -= h
        num = (loss(Pp) - loss(Pm)) / (2 * h)
        assert abs(num - G[0, 0, lane]) <= 1e-4 * abs(num) + 1e-9, (lane, num, G[0, 0, lane])
