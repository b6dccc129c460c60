"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle stage against a closed form, a library routine,
brute force on a small input, an identity or central finite differences, so
that a dropped term, wrong sign or transposed operand in the oracle fails here.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.ndimage
import scipy.special

import oracle
import scenes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ SH basis
def _real_sh_scipy(l, m, d):
    """Real SH from scipy's complex Y_l^m (Condon-Shortley phase included):
    sqrt2 Re Y_l^m for m > 0, sqrt2 Im Y_l^|m| for m < 0, Y_l^0 for m = 0."""
    x, y, z = d
    theta = math.acos(max(-1.0, min(1.0, z)))  # polar
    phi = math.atan2(y, x)  # azimuth
    Yc = scipy.special.sph_harm_y(l, abs(m), theta, phi)
    if m > 0:
        return math.sqrt(2.0) * Yc.real
    if m < 0:
        return math.sqrt(2.0) * Yc.imag
    return Yc.real


def test_sh_basis_matches_scipy_complex_harmonics():
    rng = np.random.default_rng(1)
    for _ in range(25):
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        Y, _ = oracle.sh_basis(d)
        for l in range(4):
            for m in range(-l, l + 1):
                k = l * l + l + m
                assert Y[k] == pytest.approx(_real_sh_scipy(l, m, d), abs=1e-12), (l, m)


def test_sh_basis_orthonormal_by_quadrature():
    # Gauss-Legendre in cos(theta) x uniform phi: exact for degree <= 6 products
    nt, npf = 12, 24
    xs, ws = np.polynomial.legendre.leggauss(nt)
    G = np.zeros((16, 16))
    for ct, wt in zip(xs, ws):
        st = math.sqrt(1 - ct * ct)
        for j in range(npf):
            ph = 2 * math.pi * j / npf
            Y, _ = oracle.sh_basis(np.array([st * math.cos(ph), st * math.sin(ph), ct]))
            G += wt * (2 * math.pi / npf) * np.outer(Y, Y)
    assert np.allclose(G, np.eye(16), atol=1e-12)


def test_sh_gradient_matches_central_differences():
    rng = np.random.default_rng(2)
    for _ in range(10):
        d = rng.standard_normal(3)
        d /= np.linalg.norm(d)
        _, dY = oracle.sh_basis(d)
        h = 1e-6
        for ax in range(3):
            e = np.zeros(3)
            e[ax] = h
            num = (oracle.sh_basis(d + e)[0] - oracle.sh_basis(d - e)[0]) / (2 * h)
            assert np.allclose(dY[:, ax], num, atol=1e-8)


# ------------------------------------------------------------------ closed form, one isotropic Gaussian
@pytest.mark.parametrize("logs,logit,sh0", [(-2.0, 0.3, 0.7), (-3.0, 2.5, 1.4), (-1.5, -1.0, 0.2)])
def test_single_isotropic_gaussian_closed_form(logs, logit, sh0):
    W = H = 128
    f = 140.0
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), W, H, f)
    P = np.zeros((15, 1, 4), np.float32)
    P[1, 0, :3] = logs
    P[0, 0, 3] = logit
    q = np.array([0.3, -0.5, 0.7, 0.2])
    P[2, 0] = q / np.linalg.norm(q)  # any rotation of an isotropic Gaussian
    P[3, 0, 0] = P[3, 0, 1] = P[3, 0, 2] = sh0
    s = math.exp(np.float32(logs))
    o = 1.0 / (1.0 + math.exp(-float(np.float32(logit))))
    var = (f * s / 4.0) ** 2 + 0.3
    pr = oracle.project(P, cam)
    assert pr["uvzo"][0, :3] == pytest.approx([64.0, 64.0, 4.0])
    assert pr["conic"][0] == pytest.approx([1 / var, 0.0, 1 / var], rel=1e-12, abs=1e-14)
    assert pr["radius"][0] == math.ceil(3 * math.sqrt(var))
    colour = 0.5 / math.sqrt(math.pi) * float(np.float32(sh0)) + 0.5
    assert pr["rgb"][0] == pytest.approx([colour] * 3, rel=1e-12)
    img = oracle.render_view(P, cam)
    r = pr["radius"][0]
    t0, t1 = max(0, (64 - r) // 16), min(8, (64 + r) // 16 + 1)
    expect = np.zeros((H, W))
    for py in range(H):
        for px in range(W):
            if not (t0 <= px // 16 < t1 and t0 <= py // 16 < t1):
                continue
            rho2 = (px + 0.5 - 64) ** 2 + (py + 0.5 - 64) ** 2
            a = min(0.99, o * math.exp(-rho2 / (2 * var)))
            if np.float32(a) >= np.float32(1 / 255):
                expect[py, px] = colour * a
    for c in range(3):
        assert np.allclose(img[c], expect, atol=1e-12)


# ------------------------------------------------------------------ brute-force compositing
def _brute_force_image(pr, W, H):
    """Every pixel: all r > 0 Gaussians whose tile square covers the pixel's tile,
    sorted by (fp32 depth, index), composited front to back.  Also counts, per pixel, the
    entries evaluated (through the one that ends the walk, else all) and accumulated."""
    N = pr["radius"].shape[0]
    u = pr["uvzo"][:, 0].astype(np.float32).astype(np.float64)
    v = pr["uvzo"][:, 1].astype(np.float32).astype(np.float64)
    z32 = pr["uvzo"][:, 2].astype(np.float32)
    r = pr["radius"]
    tx, ty = (W + 15) // 16, (H + 15) // 16
    x0 = np.clip(np.floor((u - r) / 16), 0, tx)
    x1 = np.clip(np.floor((u + r) / 16) + 1, 0, tx)
    y0 = np.clip(np.floor((v - r) / 16), 0, ty)
    y1 = np.clip(np.floor((v + r) / 16) + 1, 0, ty)
    img = np.zeros((3, H, W))
    Tf = np.ones((H, W))
    n_eval = np.zeros((H, W), np.uint32)
    n_used = np.zeros((H, W), np.uint32)
    for py in range(H):
        for px in range(W):
            tX, tY = px // 16, py // 16
            sel = np.nonzero((r > 0) & (x0 <= tX) & (tX < x1) & (y0 <= tY) & (tY < y1))[0]
            order = sorted(sel.tolist(), key=lambda i: (float(z32[i]), i))
            T = 1.0
            C = np.zeros(3)
            n_eval[py, px] = len(order)
            for pos, i in enumerate(order):
                dx = px + 0.5 - pr["uvzo"][i, 0]
                dy = py + 0.5 - pr["uvzo"][i, 1]
                A, B, Cc = pr["conic"][i]
                power = -0.5 * (A * dx * dx + Cc * dy * dy) - B * dx * dy
                if np.float32(power) > 0:
                    continue
                a = pr["uvzo"][i, 3] * math.exp(power)
                if np.float32(a) > np.float32(0.99):
                    a = float(np.float32(0.99))
                if np.float32(a) < np.float32(1.0 / 255.0):
                    continue
                Tn = T * (1 - a)
                if np.float32(Tn) < np.float32(1e-4):
                    n_eval[py, px] = pos + 1
                    break
                C += pr["rgb"][i] * a * T
                T = Tn
                n_used[py, px] += 1
            img[:, py, px] = C
            Tf[py, px] = T
    return img, Tf, n_eval, n_used


@pytest.mark.parametrize("seed,n", [(3, 40), (4, 150)])
def test_tiled_compositing_equals_brute_force(seed, n):
    P, cam = scenes.tiny_scene(n, seed, width=48, height=40, focal=50.0, logscale=(-2.5, -1.2),
                               opacity=(0.0, 3.0))
    pr = oracle.project(P, cam)
    assert (pr["radius"] > 0).sum() > n // 2
    keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], cam.width, cam.height)
    img, T, nc, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, cam.width, cam.height)
    ref, Tref, eval_ref, used_ref = _brute_force_image(pr, cam.width, cam.height)
    assert np.allclose(img, ref, atol=1e-12)
    assert np.allclose(T, Tref, atol=1e-12)
    n_eval, n_used = oracle.render_counts(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, cam.width, cam.height)
    assert np.array_equal(n_eval, eval_ref) and np.array_equal(n_used, used_ref)
    assert (n_used <= nc).all() and (nc <= n_eval).all()
    tx = (cam.width + 15) // 16
    ys, xs = np.mgrid[0:cam.height, 0:cam.width]
    lens = (ranges[:, 1] - ranges[:, 0])[(ys // 16) * tx + xs // 16]
    assert (n_eval <= lens).all()
    if seed == 4:
        assert (n_eval < lens).any()  # some walks end at the transmittance floor
    assert (n_used < nc).any()  # some entries are skipped before a pixel's last accumulated one


def test_binning_matches_python_stable_sort():
    P = scenes.make_params(0)
    cam = scenes.make_cameras(0)[0]
    pr = oracle.project(P, cam)
    keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], cam.width, cam.height)
    inst = []
    tx = cam.tiles_x
    for i in range(P.shape[1]):
        if pr["radius"][i] <= 0:
            continue
        x0, y0, x1, y1 = pr["rect"][i]
        zb = int(np.float32(pr["uvzo"][i, 2]).view(np.uint32))
        for ty in range(y0, y1):
            for tX in range(x0, x1):
                inst.append((((ty * tx + tX) << 32) | zb, i))
    inst = sorted(inst, key=lambda e: e[0])  # Python's sort is stable
    assert len(inst) == len(keys) == int(pr["tiles"].sum())
    assert [e[0] for e in inst] == keys.tolist()
    assert [e[1] for e in inst] == vals.tolist()
    tiles = keys >> np.uint64(32)
    for t in range(cam.n_tiles):
        idx = np.nonzero(tiles == t)[0]
        if idx.size:
            assert tuple(ranges[t]) == (idx[0], idx[-1] + 1)
        else:
            assert tuple(ranges[t]) == (0, 0)


# ------------------------------------------------------------------ compositing invariants
def test_compositing_invariants_config0():
    P = scenes.make_params(0)
    cam = scenes.make_cameras(0)[0]
    pr = oracle.project(P, cam)
    keys, vals, ranges = oracle.bin_sort(pr["uvzo"], pr["radius"], cam.width, cam.height)
    white = np.ones_like(pr["rgb"])
    img, T, nc, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], white, vals, ranges, cam.width, cam.height)
    # sum of weights + final transmittance = 1 (telescoping product)
    assert np.allclose(img[0] + T, 1.0, atol=1e-12)
    assert (T >= 1e-4 * (1 - 1e-6)).all() and (T <= 1.0).all()
    lens = (ranges[:, 1] - ranges[:, 0]).reshape(cam.tiles_y, cam.tiles_x)
    per_px = np.repeat(np.repeat(lens, 16, 0), 16, 1)[: cam.height, : cam.width]
    assert (nc <= per_px).all()
    # alpha per Gaussian never exceeds 0.99: a single Gaussian leaves T >= 0.01
    one = np.zeros_like(vals)
    one_ranges = np.zeros_like(ranges)
    r0 = int(np.argmax(lens.ravel()))
    one[0] = vals[ranges[r0, 0]]
    one_ranges[r0] = (0, 1)
    img1, T1, _, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], white, one, one_ranges, cam.width, cam.height)
    assert T1.min() >= 0.01 - 1e-12


# ------------------------------------------------------------------ finite differences of the whole step
def _fd_scene(seed, n=6):
    P, cam = scenes.tiny_scene(n, seed, width=32, height=32, focal=40.0)
    rng = np.random.default_rng(seed + 100)
    tgt = rng.uniform(0.0, 1.0, size=(1, 3, 32, 32))
    return P.astype(np.float64), cam, tgt


@pytest.mark.parametrize("seed", [11, 12])
def test_gradients_match_central_differences(seed):
    P, cam, tgt = _fd_scene(seed)
    res = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)
    G = res["grads"]
    rng = np.random.default_rng(seed)
    checked = 0
    for i in range(P.shape[1]):
        for plane in range(15):
            for lane in range(4):
                if plane == 1 and lane == 3:
                    continue
                if plane >= 3 and rng.uniform() > 0.35:
                    continue  # sample of the SH coefficients
                h = 1e-5 * max(1.0, abs(P[plane, i, lane]))
                Pp = P.copy()
                Pp[plane, i, lane] += h
                Pm = P.copy()
                Pm[plane, i, lane] -= h
                lp = oracle.step(Pp, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)["loss"]
                lm = oracle.step(Pm, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)["loss"]
                num = (lp - lm) / (2 * h)
                ana = G[plane, i, lane]
                # relative 1e-4, with an absolute floor for the double-precision
                # rounding of the loss divided by h (about 1e-16 / 1e-5)
                assert abs(num - ana) <= 1e-4 * abs(num) + 1e-9, (i, plane, lane, num, ana)
                checked += 1
    assert checked > 100


# ------------------------------------------------------------------ loss
def _ssim_scipy(x, y):
    h = np.exp(-((np.arange(11) - 5.0) ** 2) / (2 * 1.5 ** 2))
    h /= h.sum()
    w = np.outer(h, h)
    conv = lambda a: scipy.ndimage.correlate(a, w, mode="constant", cval=0.0)
    C1, C2 = 0.01 ** 2, 0.03 ** 2
    out = []
    for c in range(3):
        mx, my = conv(x[c]), conv(y[c])
        sxx = conv(x[c] * x[c]) - mx * mx
        syy = conv(y[c] * y[c]) - my * my
        sxy = conv(x[c] * y[c]) - mx * my
        out.append(((2 * mx * my + C1) * (2 * sxy + C2)) / ((mx * mx + my * my + C1) * (sxx + syy + C2)))
    return np.mean(out)


def test_loss_matches_scipy_window_sums():
    rng = np.random.default_rng(5)
    x = rng.uniform(size=(3, 23, 31))
    y = rng.uniform(size=(3, 23, 31))
    val, _ = oracle.loss(x, y, grad=False)
    ref = 0.8 * np.mean(np.abs(x - y)) + 0.2 * (1 - _ssim_scipy(x, y))
    assert val == pytest.approx(ref, rel=1e-12)
    val2, _ = oracle.loss(x, y, scale=0.25, grad=False)
    assert val2 == pytest.approx(0.25 * ref, rel=1e-12)


def test_loss_identity_and_gradient():
    rng = np.random.default_rng(6)
    x = rng.uniform(size=(3, 17, 19))
    val, d = oracle.loss(x, x)
    assert abs(val) < 1e-14
    assert np.abs(d).max() < 1e-14
    y = rng.uniform(size=(3, 17, 19))
    val, d = oracle.loss(x, y, scale=0.5)
    h = 1e-6
    for _ in range(40):
        c, i, j = rng.integers(3), rng.integers(17), rng.integers(19)
        xp = x.copy()
        xp[c, i, j] += h
        xm = x.copy()
        xm[c, i, j] -= h
        num = (oracle.loss(xp, y, scale=0.5, grad=False)[0] - oracle.loss(xm, y, scale=0.5, grad=False)[0]) / (2 * h)
        assert d[c, i, j] == pytest.approx(num, rel=1e-5, abs=1e-11)


# ------------------------------------------------------------------ Adam
def test_batch_scaling_rule_golden():
    with open(os.path.join(GOLDEN, "batch_scaling.json")) as fh:
        g = json.load(fh)
    for case in g["cases"]:
        b = case["batch"]
        # t = 1: m_hat = g and v_hat = g^2, so the step is lr' * sign(g)
        P = np.zeros((15, 1, 4))
        G = np.zeros((15, 1, 4))
        G[0, 0, 0] = 0.25
        G[0, 0, 1] = -3.0
        p, gr, m, v = oracle.sparse_adam(P, G, np.zeros_like(P), np.zeros_like(P), [0], g["lr"], g["beta1"],
                                         g["beta2"], 1e-15, b, 1)
        assert p[0, 0, 0] == pytest.approx(-case["lr_scaled"], rel=1e-12)
        assert p[0, 0, 1] == pytest.approx(case["lr_scaled"], rel=1e-12)
        assert m[0, 0, 0] == pytest.approx((1 - case["beta1_scaled"]) * 0.25, rel=1e-12)
        assert v[0, 0, 1] == pytest.approx((1 - case["beta2_scaled"]) * 9.0, rel=1e-12)
        assert (gr == 0).all()


def test_adam_two_steps_closed_form_and_untouched_rows():
    rng = np.random.default_rng(7)
    N = 5
    P = rng.standard_normal((15, N, 4))
    G1 = rng.standard_normal((15, N, 4))
    lr, b1, b2, eps, B = 1e-2, 0.9, 0.999, 1e-15, 2
    p1, g1, m1, v1 = oracle.sparse_adam(P, G1, np.zeros_like(P), np.zeros_like(P), [1, 3], lr, b1, b2, eps, B, 1)
    for i in (0, 2, 4):  # not listed: bit-for-bit unchanged, gradient kept
        assert (p1[:, i] == P[:, i]).all() and (m1[:, i] == 0).all() and (g1[:, i] == G1[:, i]).all()
    G2 = rng.standard_normal((15, N, 4))
    p2, _, m2, v2 = oracle.sparse_adam(p1, G2, m1, v1, [1, 3], lr, b1, b2, eps, B, 2)
    bb1, bb2, lrb = b1 ** B, b2 ** B, lr * math.sqrt(B)
    for i in (1, 3):
        m_ = bb1 * (1 - bb1) * G1[:, i] + (1 - bb1) * G2[:, i]
        v_ = bb2 * (1 - bb2) * G1[:, i] ** 2 + (1 - bb2) * G2[:, i] ** 2
        exp_p = p1[:, i] - lrb * (m_ / (1 - bb1 ** 2)) / (np.sqrt(v_ / (1 - bb2 ** 2)) + eps)
        assert np.allclose(m2[:, i], m_, rtol=1e-13)
        assert np.allclose(v2[:, i], v_, rtol=1e-13)
        assert np.allclose(p2[:, i], exp_p, rtol=1e-12, atol=1e-15)


def test_identical_views_batch_gradient_equals_single_view():
    P, cam, tgt = _fd_scene(21)
    one = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt, do_adam=False)
    four = oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam] * 4, np.repeat(tgt, 4, 0), do_adam=False)
    assert four["loss"] == pytest.approx(one["loss"], rel=1e-12)
    assert np.allclose(four["grads"], one["grads"], rtol=1e-11, atol=1e-15)


# ------------------------------------------------------------------ visible sets
def test_visible_sets_against_python_sets():
    rng = np.random.default_rng(8)
    B, N = 6, 500
    radii = np.where(rng.uniform(size=(B, N)) < np.linspace(0.05, 0.8, B)[:, None], rng.integers(1, 9, (B, N)), 0)
    radii[4] = 0  # an empty view
    off, ind, uni, inter, jac = oracle.visible_sets(radii.astype(np.int32))
    sets = [set(np.nonzero(radii[b] > 0)[0].tolist()) for b in range(B)]
    for b in range(B):
        assert ind[off[b]:off[b + 1]].tolist() == sorted(sets[b])
    assert uni.tolist() == sorted(set().union(*sets))
    for i in range(B):
        for j in range(B):
            n = len(sets[i] & sets[j])
            un = len(sets[i] | sets[j])
            assert inter[i, j] == n
            assert jac[i, j] == (np.float32(n / un) if un else 0.0)
    assert (inter == inter.T).all()
    assert jac[4, 4] == 0.0 and jac[0, 0] == 1.0
