"""Seeded synthetic scenes and cameras for the 3D Gaussian Splatting training step.

This module only draws inputs: Gaussian parameter records, pinhole cameras and
a per-view perturbation seed.  It holds none of the splatting arithmetic, so the
CUDA path and the CPU oracle can both take their inputs from it.

Parameter record (Grendel-GS notes, "背景知识" parameter table): position (3),
scale (3), rotation quaternion (4), opacity (1) and 48 SH coefficients, 59 floats
per Gaussian.  They are stored as 15 float4 planes, plane-major, shape
``[15, N, 4]`` float32:

* plane 0  = (x, y, z, opacity logit)
* plane 1  = (log s0, log s1, log s2, 0)
* plane 2  = (qw, qx, qy, qz)
* planes 3..14 = the 48 SH coefficients sh[k][c] (k = 0..15, c = r, g, b)
  flattened as 3*k + c, four per plane.

Cameras use OpenCV axes (x right, y down, z forward); ``R`` maps world to
camera, ``p_cam = R @ p + t``.  World -y is "up" for the generated orbits.

All draws use numpy's PCG64 with fixed seeds: parameters from ``seed``, cameras
from ``1000 + seed`` and the target-render jitter from ``2000 + seed``.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

TILE = 16
N_PLANES = 15


@dataclasses.dataclass
class Camera:
    R: np.ndarray  # (3, 3) float32, world -> camera rows
    t: np.ndarray  # (3,) float32
    fx: float
    fy: float
    cx: float
    cy: float
    znear: float
    width: int
    height: int

    @property
    def tiles_x(self) -> int:
        return (self.width + TILE - 1) // TILE

    @property
    def tiles_y(self) -> int:
        return (self.height + TILE - 1) // TILE

    @property
    def n_tiles(self) -> int:
        return self.tiles_x * self.tiles_y


@dataclasses.dataclass
class SceneConfig:
    name: str
    n: int
    width: int
    height: int
    focal: float
    batch: int
    n_views: int
    layout: str
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-15
    znear: float = 0.2
    w_l1: float = 0.8
    w_ssim: float = 0.2
    jitter: float = 0.02


# The five workloads: sizes, layouts, resolutions and batch sizes of the
# published scales (a 2K-Gaussian toy, an object scene, an unbounded scene, the
# one-GPU limit of about 11M Gaussians, and a 4K / 40M scene).
CONFIGS = {
    0: SceneConfig("tiny-2k-128px", 2048, 128, 128, 140.0, 1, 1, "cube"),
    1: SceneConfig("object-300k-1236x820", 300_000, 1236, 820, 1100.0, 4, 64, "clusters64"),
    2: SceneConfig("unbounded-3m-1237x822", 3_000_000, 1237, 822, 1100.0, 8, 200, "core_shell"),
    3: SceneConfig("city-11m-1920x1080", 11_000_000, 1920, 1080, 0.89 * 1920, 4, 64, "city16"),
    4: SceneConfig("city-40m-3840x2160", 40_000_000, 3840, 2160, 0.89 * 3840, 16, 64, "city32"),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _means(layout: str, n: int, rng: np.random.Generator) -> np.ndarray:
    if layout == "cube":
        return rng.uniform(-1.0, 1.0, size=(n, 3))
    if layout == "clusters64":
        k = 64
        # cluster centres uniform in the ball of radius 1.4
        d = rng.standard_normal((k, 3))
        d /= np.linalg.norm(d, axis=1, keepdims=True)
        centres = d * (1.4 * rng.uniform(0.0, 1.0, size=(k, 1)) ** (1.0 / 3.0))
        sig = rng.uniform(0.05, 0.3, size=(k, 3))
        # random cluster orientations: orthonormal factor of a Gaussian matrix
        rot = np.stack([np.linalg.qr(rng.standard_normal((3, 3)))[0] for _ in range(k)])
        lab = rng.integers(0, k, size=n)
        out = np.empty((n, 3))
        todo = np.arange(n)
        while todo.size:
            z = rng.standard_normal((todo.size, 3)) * sig[lab[todo]]
            p = centres[lab[todo]] + np.einsum("nij,nj->ni", rot[lab[todo]], z)
            ok = np.linalg.norm(p, axis=1) <= 2.0
            out[todo[ok]] = p[ok]
            todo = todo[~ok]
        return out
    if layout == "core_shell":
        n_core = int(round(0.8 * n))
        d = rng.standard_normal((n, 3))
        d /= np.linalg.norm(d, axis=1, keepdims=True)
        r = np.empty(n)
        r[:n_core] = 1.5 * rng.uniform(0.0, 1.0, size=n_core) ** (1.0 / 3.0)
        r[n_core:] = np.exp(rng.uniform(math.log(1.5), math.log(50.0), size=n - n_core))
        return d * r[:, None]
    if layout in ("city16", "city32"):
        g = 16 if layout == "city16" else 32
        pitch = 1.5
        h = rng.uniform(0.5, 3.0, size=g * g)
        cell = rng.integers(0, g * g, size=n)
        cx = (cell % g - (g - 1) / 2.0) * pitch
        cz = (cell // g - (g - 1) / 2.0) * pitch
        u = rng.uniform(0.0, 1.0, size=(n, 3))
        x = cx + (u[:, 0] - 0.5)
        z = cz + (u[:, 2] - 0.5)
        y = -u[:, 1] * h[cell]  # boxes rise toward world -y
        return np.stack([x, y, z], axis=1)
    raise ValueError(layout)


def make_params(cfg: SceneConfig | int, seed: int | None = None, n: int | None = None) -> np.ndarray:
    """Draw the ``[15, N, 4]`` float32 parameter planes of one scene.

    Draw order (fixed): means, log-scales U[-4.5,-2.5], quaternions N(0, I4)
    normalised, opacity logits N(0,1), SH DC N(0.5, 0.2), SH rest N(0, 0.05).
    """
    if isinstance(cfg, int):
        if seed is None:
            seed = cfg
        cfg = CONFIGS[cfg]
    if seed is None:
        seed = 0
    n = cfg.n if n is None else n
    rng = _rng(seed)
    P = np.zeros((N_PLANES, n, 4), dtype=np.float32)
    P[0, :, :3] = _means(cfg.layout, n, rng)
    P[1, :, :3] = rng.uniform(-4.5, -2.5, size=(n, 3))
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    P[2] = q
    del q
    P[0, :, 3] = rng.standard_normal(n)
    # the SH coefficients, drawn in blocks of Gaussians (the same stream as one draw of all of
    # them) so that no float64 copy of the whole [n, 48] array is ever held
    sh = P[3:].transpose(1, 0, 2).reshape(n, 48) if n else np.zeros((0, 48), np.float32)
    chunk = 1 << 20
    for a in range(0, n, chunk):
        sh[a:a + chunk, :3] = rng.normal(0.5, 0.2, size=(min(chunk, n - a), 3))
    for a in range(0, n, chunk):
        sh[a:a + chunk, 3:] = rng.normal(0.0, 0.05, size=(min(chunk, n - a), 45))
    P[3:] = sh.reshape(n, 12, 4).transpose(1, 0, 2)
    return P


def jitter_means(params: np.ndarray, sigma: float, seed: int) -> np.ndarray:
    """Copy of ``params`` with every mean moved by N(0, sigma^2) per axis."""
    rng = _rng(seed)
    out = params.copy()
    n = params.shape[1]
    out[0, :, :3] += rng.normal(0.0, sigma, size=(n, 3)).astype(np.float32)
    return out


def look_at(eye, target, width, height, focal, znear=0.2) -> Camera:
    """Pinhole camera at ``eye`` looking at ``target`` with world -y as up."""
    eye = np.asarray(eye, dtype=np.float64)
    target = np.asarray(target, dtype=np.float64)
    zc = target - eye
    zc /= np.linalg.norm(zc)
    xc = np.cross(zc, np.array([0.0, -1.0, 0.0]))
    xc /= np.linalg.norm(xc)
    yc = np.cross(zc, xc)
    R = np.stack([xc, yc, zc])
    t = -R @ eye
    return Camera(R.astype(np.float32), t.astype(np.float32), float(focal), float(focal),
                  width / 2.0, height / 2.0, znear, width, height)


def make_cameras(cfg: SceneConfig | int, seed: int | None = None) -> list[Camera]:
    """All training views of a workload (seed ``1000 + k`` by convention)."""
    if isinstance(cfg, int):
        if seed is None:
            seed = 1000 + cfg
        cfg = CONFIGS[cfg]
    if seed is None:
        seed = 1000
    rng = _rng(seed)
    W, H, f = cfg.width, cfg.height, cfg.focal
    cams = []
    if cfg.layout == "cube":
        cams.append(look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), W, H, f, cfg.znear))
        return cams
    phase = rng.uniform(0.0, 2 * math.pi)
    for k in range(cfg.n_views):
        th = phase + 2 * math.pi * k / cfg.n_views
        if cfg.layout == "clusters64":
            eye = (5.0 * math.cos(th), 0.0, 5.0 * math.sin(th))
            tgt = (0.0, 0.0, 0.0)
        elif cfg.layout == "core_shell":
            eye = (4.0 * math.cos(th), 0.0, 4.0 * math.sin(th))
            # every 4th view looks up so its top half sees only the sparse shell
            tgt = (0.0, -1.5, 0.0) if k % 4 == 3 else (0.0, 0.0, 0.0)
        else:
            rad, hgt = (16.0, 8.0) if cfg.layout == "city16" else (32.0, 16.0)
            eye = (rad * math.cos(th), -hgt, rad * math.sin(th))
            tgt = (0.0, -0.5, 0.0)
        cams.append(look_at(eye, tgt, W, H, f, cfg.znear))
    return cams


def batch_views(cfg: SceneConfig, step: int) -> list[int]:
    """View indices of batch ``step``: consecutive views around the orbit."""
    return [((step * cfg.batch) + b) % cfg.n_views for b in range(cfg.batch)]


def synthetic_targets(batch: int, width: int, height: int, seed: int) -> np.ndarray:
    """Seeded target images [batch, 3, H, W] float32 in [0.1, 0.9]: per channel, a sum of four
    plane waves of random direction, wavelength (8 to 200 px) and phase, rescaled.  Stands in
    for the photographs a training step compares against where rendering a target is too
    costly for the CPU oracle."""
    rng = _rng(seed)
    y, x = np.mgrid[0:height, 0:width].astype(np.float32)
    out = np.empty((batch, 3, height, width), np.float32)
    for b in range(batch):
        for c in range(3):
            acc = np.zeros((height, width), np.float32)
            for _ in range(4):
                th = rng.uniform(0.0, 2 * math.pi)
                lam = math.exp(rng.uniform(math.log(8.0), math.log(200.0)))
                ph = rng.uniform(0.0, 2 * math.pi)
                k = 2 * math.pi / lam
                acc += np.cos(np.float32(k * math.cos(th)) * x + np.float32(k * math.sin(th)) * y + np.float32(ph))
            out[b, c] = 0.5 + 0.1 * acc
    return out


def tiny_scene(n: int, seed: int, width: int = 32, height: int = 32, focal: float = 40.0,
               spread: float = 0.6, logscale=(-2.2, -1.6), opacity=(0.1, 1.2)):
    """Few-Gaussian scene for finite-difference and brute-force checks.

    Means lie in a small box in front of a camera at (0, 0, -4); scales and
    opacity logits are kept in ranges whose alphas stay away from the 1/255
    skip and the 0.99 clamp.
    """
    rng = _rng(seed)
    P = np.zeros((N_PLANES, n, 4), dtype=np.float32)
    P[0, :, :2] = rng.uniform(-spread, spread, size=(n, 2))
    P[0, :, 2] = rng.uniform(-0.5, 0.5, size=n)
    P[0, :, 3] = rng.uniform(opacity[0], opacity[1], size=n) * rng.choice([-1.0, 1.0], size=n)
    P[1, :, :3] = rng.uniform(logscale[0], logscale[1], size=(n, 3))
    q = rng.standard_normal((n, 4))
    P[2] = q / np.linalg.norm(q, axis=1, keepdims=True)
    sh = np.concatenate([rng.normal(0.5, 0.2, size=(n, 3)), rng.normal(0.0, 0.08, size=(n, 45))], axis=1)
    P[3:] = sh.astype(np.float32).reshape(n, 12, 4).transpose(1, 0, 2)
    cam = look_at((0.0, 0.0, -4.0), (0.0, 0.0, 0.0), width, height, focal)
    return P, cam
