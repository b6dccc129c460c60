"""Pins of the oracle's forward projection for anisotropic, rotated, off-axis Gaussians.

The 2-D covariance the oracle reports (through its conic, the inverse of the dilated
covariance) is checked against routes that share nothing with the oracle's code:

* the rotation of a unit quaternion (w, x, y, z) from ``scipy.spatial.transform``
  (scalar-last order there);
* the 3-D covariance as a direct numpy product R diag(s^2) R^T;
* the perspective Jacobian as central differences of the pinhole map
  (fx x / z + cx, fy y / z + cy) at the camera-space mean, evaluated where the
  field-of-view clamp puts it (x/z and y/z limited to 1.3 tan(fov / 2));
* screen positions as the pinhole map itself;
* hand-worked closed forms (axis-aligned scales off the axis, quarter turns that
  swap scale axes, a mean beyond the clamp);
* the view-dependent colour against real harmonics built from scipy's complex ones,
  with the direction taken from the camera centre to the mean (odd degrees change sign
  between two opposite cameras).

Grendel-GS notes, 训练流程 "高斯变换" (3-D Gaussian to screen position, footprint and
colour); the readings of the camera, the EWA Jacobian, its clamp and the low-pass 0.3
are the ones the oracle's header states.
"""
import math

import numpy as np
import pytest
from scipy.spatial.transform import Rotation

import oracle
import scenes
from test_oracle_pins import _real_sh_scipy

F32 = np.float32


def _f64(a):
    return np.asarray(a, np.float32).astype(np.float64)


def _params(mu, logs, q, logit=1.0, sh=None):
    """One Gaussian as the [15, 1, 4] float32 planes (values exactly representable are used
    where a closed form needs them)."""
    P = np.zeros((15, 1, 4), np.float32)
    P[0, 0, :3] = mu
    P[0, 0, 3] = logit
    P[1, 0, :3] = logs
    P[2, 0] = q
    if sh is not None:
        P[3:, 0] = np.asarray(sh, np.float32).reshape(12, 4)
    return P


def _cov_from_conic(conic):
    A, B, C = conic
    return np.linalg.inv(np.array([[A, B], [B, C]]))


def _pinhole(cam, p):
    return np.array([cam.fx * p[0] / p[2] + cam.cx, cam.fy * p[1] / p[2] + cam.cy])


def _jacobian_fd(cam, p, h=1e-6):
    J = np.zeros((2, 3))
    for k in range(3):
        e = np.zeros(3)
        e[k] = h * max(1.0, abs(p[k]))
        J[:, k] = (_pinhole(cam, p + e) - _pinhole(cam, p - e)) / (2 * e[k])
    return J


def _expected(P, cam):
    """Screen position and dilated 2-D covariance from scipy / numpy / differences."""
    mu = _f64(P[0, 0, :3])
    s = np.exp(_f64(P[1, 0, :3]))
    w, x, y, z = _f64(P[2, 0])
    Rq = Rotation.from_quat([x, y, z, w]).as_matrix()  # normalises the quaternion itself
    Sigma = Rq @ np.diag(s * s) @ Rq.T
    Rw, t = _f64(cam.R), _f64(cam.t)
    pc = Rw @ mu + t
    lim = np.array([1.3 * (cam.width / 2.0) / cam.fx, 1.3 * (cam.height / 2.0) / cam.fy])
    ratio = np.clip(pc[:2] / pc[2], -lim, lim)
    p_j = np.array([ratio[0] * pc[2], ratio[1] * pc[2], pc[2]])  # where the Jacobian is taken
    J = _jacobian_fd(cam, p_j)
    cov = J @ (Rw @ Sigma @ Rw.T) @ J.T + 0.3 * np.eye(2)
    return _pinhole(cam, pc), pc[2], cov


def _generic_camera(W=160, H=120, f=150.0, eye=(2.6, -1.3, -3.1), target=(0.2, 0.1, 0.05)):
    return scenes.look_at(eye, target, W, H, f)


@pytest.mark.parametrize("seed", range(6))
def test_anisotropic_rotated_off_axis_against_scipy_and_differences(seed):
    rng = np.random.default_rng(700 + seed)
    cam = _generic_camera()
    checked = 0
    for _ in range(40):
        q = rng.standard_normal(4)
        mu = rng.uniform(-0.8, 0.8, 3)
        logs = rng.uniform(-3.0, -1.2, 3)
        P = _params(mu, logs, q)
        pr = oracle.project(P, cam)
        if pr["radius"][0] <= 0:
            continue
        uv, depth, cov = _expected(P, cam)
        assert pr["uvzo"][0, :2] == pytest.approx(uv, rel=1e-12, abs=1e-9)
        assert pr["uvzo"][0, 2] == pytest.approx(depth, rel=1e-12)
        got = _cov_from_conic(pr["conic"][0])
        assert np.allclose(got, cov, rtol=1e-7, atol=1e-9 * np.abs(cov).max()), (got, cov)
        lam = np.linalg.eigvalsh(cov).max()
        r3 = 3.0 * math.sqrt(lam)
        if abs(r3 - round(r3)) > 1e-6:
            assert pr["radius"][0] == math.ceil(r3)
        o = 1.0 / (1.0 + math.exp(-float(P[0, 0, 3])))
        assert pr["uvzo"][0, 3] == pytest.approx(o, rel=1e-12)
        checked += 1
    assert checked >= 25


def test_axis_aligned_scales_off_axis_hand_worked():
    """Identity rotation, camera at (0, 0, -4) looking down +z (world = camera axes up to
    the translation): Sigma2D = J diag(sx^2, sy^2, sz^2) J^T + 0.3 I with
    J = [[f/z, 0, -f x/z^2], [0, f/z, -f y/z^2]], written out entry by entry."""
    W = H = 128
    f = 140.0
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), W, H, f)
    mu = np.array([0.5, -0.375, 0.25])  # exactly representable
    logs = np.array([-2.0, -1.5, -1.0])
    P = _params(mu, logs, (1.0, 0.0, 0.0, 0.0))
    sx, sy, sz = np.exp(_f64(logs))
    x, y, z = mu[0], mu[1], mu[2] + 4.0
    c00 = (f / z) ** 2 * sx ** 2 + (f * x / z ** 2) ** 2 * sz ** 2 + 0.3
    c01 = (f * x / z ** 2) * (f * y / z ** 2) * sz ** 2
    c11 = (f / z) ** 2 * sy ** 2 + (f * y / z ** 2) ** 2 * sz ** 2 + 0.3
    pr = oracle.project(P, cam)
    assert pr["radius"][0] > 0
    assert pr["uvzo"][0, 0] == pytest.approx(f * x / z + W / 2, rel=1e-14)
    assert pr["uvzo"][0, 1] == pytest.approx(f * y / z + H / 2, rel=1e-14)
    got = _cov_from_conic(pr["conic"][0])
    assert got == pytest.approx(np.array([[c00, c01], [c01, c11]]), rel=1e-12)
    assert c01 < 0  # x > 0, y < 0: the off-diagonal's sign is part of the pin


@pytest.mark.parametrize("axis,swap", [("z", (1, 0)), ("x", (0, 2))])
def test_quarter_turns_swap_scale_axes(axis, swap):
    """A 90-degree turn about z exchanges the x and y scale axes; about x it exchanges y and
    z.  On the optical axis at depth 4 the screen covariance is (f/4)^2 diag of the two
    scales that end up along world x and y, plus 0.3."""
    f = 140.0
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), 128, 128, f)
    c, s = math.cos(math.pi / 4), math.sin(math.pi / 4)
    q = (c, 0.0, 0.0, s) if axis == "z" else (c, s, 0.0, 0.0)
    logs = np.array([-2.5, -2.0, -1.5])
    P = _params((0.0, 0.0, 0.0), logs, q)
    sc = np.exp(_f64(logs))
    pr = oracle.project(P, cam)
    got = _cov_from_conic(pr["conic"][0])
    want = np.diag([(f / 4) ** 2 * sc[swap[0]] ** 2 + 0.3, (f / 4) ** 2 * sc[swap[1]] ** 2 + 0.3])
    assert np.allclose(got, want, rtol=1e-12, atol=1e-9)


@pytest.mark.parametrize("ratio", [(2.0, 0.3), (-1.8, 0.0), (0.4, 1.9), (1.7, -1.6)])
def test_mean_beyond_the_field_of_view_clamp(ratio):
    """x/z (or y/z) beyond 1.3 tan(fov/2): the Jacobian is taken at the clamped ratio while
    the screen position keeps the true one.  Closed form for an axis-aligned Gaussian on the
    config-0 camera, large enough that its footprint still reaches the image."""
    W = H = 128
    f = 140.0
    cam = scenes.look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), W, H, f)
    z = 4.0
    tan = (W / 2.0) / f
    mu = np.array([ratio[0] * tan * z, ratio[1] * tan * z, 0.0], np.float32)
    logs = np.array([0.2, 0.1, -0.3])
    P = _params(mu, logs, (1.0, 0.0, 0.0, 0.0))
    sx, sy, sz = np.exp(_f64(logs))
    x, y = float(mu[0]), float(mu[1])
    xr = float(np.clip(x / z, -1.3 * tan, 1.3 * tan))
    yr = float(np.clip(y / z, -1.3 * tan, 1.3 * tan))
    j02, j12 = -f * xr / z, -f * yr / z
    c00 = (f / z) ** 2 * sx ** 2 + j02 ** 2 * sz ** 2 + 0.3
    c01 = j02 * j12 * sz ** 2
    c11 = (f / z) ** 2 * sy ** 2 + j12 ** 2 * sz ** 2 + 0.3
    pr = oracle.project(P, cam)
    assert pr["radius"][0] > 0, "the footprint must reach the image for the pin to bite"
    assert pr["uvzo"][0, 0] == pytest.approx(f * x / z + W / 2, rel=1e-12)
    assert pr["uvzo"][0, 1] == pytest.approx(f * y / z + H / 2, rel=1e-12, abs=1e-12)
    got = _cov_from_conic(pr["conic"][0])
    assert got == pytest.approx(np.array([[c00, c01], [c01, c11]]), rel=1e-12, abs=1e-12)
    # and the unclamped Jacobian would have given something else
    assert abs(x / z) > 1.3 * tan or abs(y / z) > 1.3 * tan


def _real_basis(d):
    return np.array([_real_sh_scipy(l, m, d) for l in range(4) for m in range(-l, l + 1)])


@pytest.mark.parametrize("k", [1, 2, 3, 9, 12, 15])
def test_odd_degree_colour_from_two_opposite_cameras(k):
    """One odd-degree coefficient: seen from eye e and from -e the view directions
    d = (mu - campos)/|mu - campos| are opposite, so the colour moves by +-sh Y_k(d)."""
    mu = np.zeros(3)
    eye = np.array([1.9, -2.3, -2.8])
    coef = np.array([0.3, -0.2, 0.25])
    sh = np.zeros((16, 3))
    sh[k] = coef
    P = _params(mu, (-2.0, -2.0, -2.0), (1.0, 0.0, 0.0, 0.0), sh=sh.ravel())
    for sgn in (1.0, -1.0):
        cam = scenes.look_at(sgn * eye, (0.0, 0.0, 0.0), 96, 96, 100.0)
        campos = -_f64(cam.R).T @ _f64(cam.t)
        d = (mu - campos) / np.linalg.norm(mu - campos)
        Yk = _real_basis(d)[k]
        pr = oracle.project(P, cam)
        assert pr["radius"][0] > 0
        assert pr["raw"][0] == pytest.approx(_f64(coef) * Yk + 0.5, rel=1e-6, abs=1e-9)
        assert abs(Yk) > 0.05  # the pin is not vacuous for this direction


def test_full_colour_against_scipy_harmonics_off_axis():
    rng = np.random.default_rng(77)
    cam = _generic_camera()
    campos = -_f64(cam.R).T @ _f64(cam.t)
    for _ in range(20):
        mu = rng.uniform(-0.7, 0.7, 3)
        sh = rng.normal(0.0, 0.3, (16, 3))
        P = _params(mu, (-2.0, -2.2, -1.9), rng.standard_normal(4), sh=sh.ravel())
        pr = oracle.project(P, cam)
        if pr["radius"][0] <= 0:
            continue
        m = _f64(P[0, 0, :3])
        d = (m - campos) / np.linalg.norm(m - campos)
        want = _f64(P[3:, 0]).reshape(16, 3).T @ _real_basis(d) + 0.5
        assert pr["raw"][0] == pytest.approx(want, rel=1e-9, abs=1e-12)
        assert pr["rgb"][0] == pytest.approx(np.maximum(want, 0.0), rel=1e-9, abs=1e-12)


def test_gradients_match_central_differences_oblique_camera_and_clamp():
    """Central differences of the whole step seen from an oblique camera (a general world ->
    camera rotation) with one Gaussian whose mean lies beyond the field-of-view clamp but
    whose footprint reaches the image, so both branches of the Jacobian's backward and the
    camera rotation's transpose are exercised."""
    W = H = 32
    P, _ = scenes.tiny_scene(5, 31, width=W, height=H, focal=40.0)
    cam = scenes.look_at((2.1, -1.4, -3.3), (0.05, -0.02, 0.1), W, H, 40.0)
    # a sixth Gaussian beyond the clamp on the camera's right, wide enough to reach the image
    Rw, t = _f64(cam.R), _f64(cam.t)
    z = 4.0
    pc = np.array([1.55 * 1.3 * (W / 2.0) / 40.0 * z, 0.1, z])
    mu_far = Rw.T @ (pc - t)
    extra = _params(mu_far, (-0.2, -0.9, -0.6), (0.9, 0.2, -0.3, 0.1), logit=0.8,
                    sh=np.r_[[0.6, 0.5, 0.4], np.zeros(45)])
    P = np.concatenate([P, extra], axis=1).astype(np.float64)
    pr = oracle.project(P, cam)
    assert pr["radius"][5] > 0
    assert abs(pc[0] / pc[2]) > 1.3 * (W / 2.0) / 40.0
    rng = np.random.default_rng(5)
    tgt = rng.uniform(0.0, 1.0, size=(1, 3, H, W))
    zeros = np.zeros_like(P)
    G = oracle.step(P, zeros, zeros, [cam], tgt, do_adam=False)["grads"]
    checked = 0
    for i in range(P.shape[1]):
        for plane in range(3):  # geometry: mean + logit, log-scales, quaternion
            for lane in range(4):
                if plane == 1 and lane == 3:
                    continue
                h = 1e-5 * max(1.0, abs(P[plane, i, lane]))
                Pp, Pm = P.copy(), P.copy()
                Pp[plane, i, lane] += h
                Pm[plane, i, lane] -= h
                lp = oracle.step(Pp, zeros, zeros, [cam], tgt, do_adam=False)["loss"]
                lm = oracle.step(Pm, zeros, zeros, [cam], tgt, do_adam=False)["loss"]
                num = (lp - lm) / (2 * h)
                assert abs(num - G[plane, i, lane]) <= 1e-4 * abs(num) + 1e-9, (i, plane, lane, num, G[plane, i, lane])
                checked += 1
    assert checked == 6 * 11
    # the clamped Gaussian's mean gradient is not zero: the pin covers its branch
    assert np.abs(G[0, 5, :3]).max() > 1e-6
