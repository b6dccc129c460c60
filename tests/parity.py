"""Helpers shared by the GPU parity tests: device transfer, oracle stage inputs, tolerances.

Tolerances (stated once, used everywhere):
  * integer / index outputs (keys, values, ranges, radii, tile counts, visible sets): exact;
  * images: |gpu - oracle| <= 1e-5 (fp32 compositing vs a double oracle);
  * gradients and updated parameters: |gpu - oracle| <= 1e-3 |oracle| + floor, floor = 1e-6
    for parameter-sized quantities; for per-pixel image gradients, whose scale is 1/(3HW),
    the floor is 1e-6 of the largest magnitude.

Discrete decisions.  An element whose discrete decision (a cull, the radius ceiling, the tile
rectangle, the 1/255 skip, the 0.99 clamp, the 1e-4 termination) lies within a relative
margin of MARGIN = 1e-5 of its threshold in the oracle can come out the other way in fp32
(the kernels' alpha carries a relative rounding error of a few 1e-6: the prescaled conic, the
quadratic form, ex2.approx).  Such elements are set aside from the exact comparison and
counted:
  * Gaussians whose projection decision can change an output (a cull; a tile rectangle that
    would add or drop a tile the Gaussian reaches with alpha >= 1/255): at most
    FLAG_FRAC_GAUSSIANS = 1e-4 of them per view;
  * Gaussians whose integer radius or tile rectangle value may differ without changing any
    image or gradient (a radius ceiling within the margin: about 2 MARGIN r3 of them, 6e-4
    at the benchmark's median r3 of 31 px and about 2e-3 where radii reach 100 px; a floor
    of the screen position within its rounding bound): at most FLAG_FRAC_VALUES = 3e-3 of
    them, each radius still within one pixel;
  * pixels: a pixel carries one decision per list entry it evaluates (about 150 on the
    300K-Gaussian benchmark view), so at the same per-decision margin about 3e-4 of its
    pixels are flagged; the bar is FLAG_FRAC_PIXELS = 1e-3 of the pixels.
A flagged pixel is still bounded by what one flipped decision can change (flag_img_bound).
The backward tests set nothing aside: the image gradient is zeroed on flagged pixels on both
sides, so a flipped decision there cannot reach any Gaussian's gradient.
"""
from __future__ import annotations

import numpy as np
import torch

MARGIN = 1e-5
FLAG_FRAC_GAUSSIANS = 1e-4
FLAG_FRAC_VALUES = 3e-3
FLAG_FRAC_PIXELS = 1e-3
IMG_ATOL = 1e-5
RTOL = 1e-3
ATOL = 1e-6


def flag_img_bound(rgb, bg=(0.0, 0.0, 0.0)) -> float:
    """Largest change one flipped compositing decision can make to a pixel.

    With c = the largest colour magnitude (Gaussian colours and background) every composite
    C_rest of the entries behind an entry lies in [0, c], so:
      * the 1/255 skip: including or skipping entry j moves the pixel by
        T_j alpha_j |c_j - C_rest| <= (1/255)(1 + MARGIN) c;
      * the 1e-4 termination: stopping before entry j or not moves it by at most
        T_j |...| <= T_j c, and a flagged stop has T_j (1 - alpha_j) ~ 1e-4 with
        alpha_j <= 0.99, so T_j <= 1e-2 (1 + MARGIN);
      * the 0.99 clamp: alpha moves by MARGIN relative: negligible.
    The bound is the largest of these."""
    c = max(float(np.abs(np.asarray(rgb)).max(initial=0.0)), float(np.abs(np.asarray(bg)).max(initial=0.0)))
    # (the entries a late stop lets through add at most T ~ 1e-4 of c more)
    return (max(1.0 / 255.0, 1e-2) * (1.0 + MARGIN) + 1e-4) * c + IMG_ATOL


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.detach().cpu().numpy()


def proj_planes_from_oracle(pr) -> np.ndarray:
    """Oracle projection (double) as the float32 [3, N, 4] planes gs_project writes."""
    n = pr["radius"].shape[0]
    P = np.zeros((3, n, 4), np.float32)
    P[0] = pr["uvzo"].astype(np.float32)
    P[1, :, :3] = pr["conic"].astype(np.float32)
    P[1, :, 3] = pr["radius"].astype(np.int32).view(np.float32)
    P[2, :, :3] = pr["rgb"].astype(np.float32)
    P[2, :, 3] = pr["tiles"].astype(np.int32).view(np.float32)
    vis = pr["radius"] > 0
    P[:, ~vis] = 0.0
    return P


def oracle_inputs_from_planes(P: np.ndarray):
    """The same float32 stage inputs, as the double arrays the oracle stage functions take."""
    uvzo = P[0].astype(np.float64)
    conic = P[1, :, :3].astype(np.float64)
    radius = P[1, :, 3].view(np.int32).copy()
    rgb = P[2, :, :3].astype(np.float64)
    return uvzo, conic, radius, rgb


def allclose_grad(gpu, ref, rtol=RTOL, atol=ATOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bad = np.abs(gpu - ref) > rtol * np.abs(ref) + atol
    return bad


def grad2d_oracle_layout(g):
    """gs_render_bwd's [n][12] record as the oracle's n x 9 (du, dv, dA, dB, dC, dop, dr, dg, db)."""
    return np.stack([g[:, 0], g[:, 1], g[:, 4], g[:, 5], g[:, 6], g[:, 2], g[:, 8], g[:, 9], g[:, 10]], axis=1)


def report(name, bad, total):
    frac = bad / max(total, 1)
    print(f"[parity] {name}: {bad} / {total} ({frac:.2e})")
    return frac
