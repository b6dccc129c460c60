"""Helpers shared by the GPU parity tests: device transfer, oracle stage inputs, tolerances.

Tolerances (stated once, used everywhere):
  * integer / index outputs (keys, values, ranges, radii, tile counts, visible sets): exact;
  * images: |gpu - oracle| <= 1e-5 (fp32 compositing vs a double oracle);
  * gradients and updated parameters: |gpu - oracle| <= 1e-3 |oracle| + floor, floor = 1e-6
    for parameter-sized quantities; for per-pixel image gradients, whose scale is 1/(3HW),
    the floor is 1e-6 of the largest magnitude;
  * elements whose discrete decision (a cull, the radius ceiling, the tile rectangle, the
    1/255 skip, the 0.99 clamp, the 1e-4 termination) lies within a relative margin of 1e-5
    of its threshold in the oracle are set aside from the exact comparison and counted; the
    count must stay below 1% of the elements (it is reported: with lists of hundreds of
    entries per pixel a few 1e-4 of the pixels carry one near-threshold decision).  A
    flagged pixel is still bounded -- it may differ by at most 4/255, the weight of a few
    entries whose alpha sits at the 1/255 skip -- and a flagged radius by one pixel.
"""
from __future__ import annotations

import numpy as np
import torch

MARGIN = 1e-5
FLAG_FRAC = 1e-2
FLAG_IMG_BOUND = 4.0 / 255.0
IMG_ATOL = 1e-5
RTOL = 1e-3
ATOL = 1e-6


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


def report(name, bad, total):
    frac = bad / max(total, 1)
    print(f"[parity] {name}: {bad} / {total} outside tolerance ({frac:.2e})")
    return frac
