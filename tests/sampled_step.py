"""Oracle side of a whole training step checked on sampled Gaussians at full size.

The CPU oracle cannot composite whole 1920x1080 or 3840x2160 views of millions of Gaussians in
seconds, but a Gaussian's screen-space gradient in a view only depends on the pixels of its
own tile rectangle, and the loss gradient of a pixel only on the image within 10 pixels of it
(two 11x11 window sums).  So for each sampled Gaussian and view the oracle:

1. finds every Gaussian that can reach the Gaussian's tile rectangle grown by one tile (a
   superset from a bound on the projected radius, then the oracle's own projection and tile
   rectangles decide membership exactly);
2. composites those tiles (per-tile lists in (depth, index) order, as the binning step
   defines them);
3. takes the loss gradient on that crop, which is exact on the inner rectangle (at least 16
   pixels from every crop edge that is not an image edge; zero padding at image edges is the
   loss's own), normalised by the full image's pixel count and the batch;
4. runs the compositing backward on the inner rectangle and the projection backward of the
   sampled Gaussian.

Test infrastructure: only the GPU parity tests call this.
"""
from __future__ import annotations

import numpy as np

import oracle

TILE = 16


def reach_superset(P, cam, boxes, also=()):
    """Indices of every Gaussian whose tile rectangle can meet one of the pixel boxes
    (x0, y0, x1, y1) of this view.  The projected radius obeys
    r = ceil(3 sqrt(lambda_max)) <= 3 sqrt((f/z)^2 (2 + xr^2 + yr^2) s_max^2 + 0.3) + 1
    (the Frobenius norm of the Jacobian bounds its spectral norm; xr, yr are the clamped
    ratios), and the rectangle spans [floor(u) - r, floor(u) + r] rounded out to tiles, so it
    stays within r + 17 pixels of (u, v)."""
    R = np.asarray(cam.R, np.float64)
    t = np.asarray(cam.t, np.float64)
    n = P.shape[1]
    keep = np.zeros(n, bool)
    limx = 1.3 * (cam.width / 2.0) / cam.fx
    limy = 1.3 * (cam.height / 2.0) / cam.fy
    for a in range(0, n, 4_000_000):
        mu = P[0, a:a + 4_000_000, :3].astype(np.float64)
        pc = mu @ R.T + t
        z = pc[:, 2]
        front = z > 0.99 * cam.znear
        zs = np.where(front, z, 1.0)
        xr = np.clip(pc[:, 0] / zs, -limx, limx)
        yr = np.clip(pc[:, 1] / zs, -limy, limy)
        smax = np.exp(P[1, a:a + 4_000_000, :3].astype(np.float64).max(axis=1))
        f = max(cam.fx, cam.fy)
        lam = (f / zs) ** 2 * (2.0 + xr * xr + yr * yr) * smax * smax + 0.3
        r = 3.0 * np.sqrt(lam) + 1.0 + TILE + 1.0
        u = cam.fx * pc[:, 0] / zs + cam.cx
        v = cam.fy * pc[:, 1] / zs + cam.cy
        hit = np.zeros(len(z), bool)
        for (x0, y0, x1, y1) in boxes:
            hit |= (u + r >= x0) & (u - r <= x1) & (v + r >= y0) & (v - r <= y1)
        keep[a:a + 4_000_000] = front & hit
    keep[np.asarray(also, np.int64)] = True
    return np.nonzero(keep)[0]


def tile_box(rect, cam, grow):
    """Tile rectangle [x0, x1) x [y0, y1) grown by `grow` tiles, clipped to the image."""
    x0, y0, x1, y1 = (int(v) for v in rect)
    return (max(0, x0 - grow), max(0, y0 - grow), min(cam.tiles_x, x1 + grow), min(cam.tiles_y, y1 + grow))


def view_gradients(P, cam, target, batch, sample):
    """Screen-space gradients (n x 9, oracle layout) of the sampled Gaussians in one view, the
    oracle's projection of them (dict) and the number of candidate Gaussians looked at."""
    W, H = cam.width, cam.height
    pr_s = oracle.project(P[:, sample], cam)
    vis = np.nonzero(pr_s["radius"] > 0)[0]
    g2d = np.zeros((len(sample), 9))
    if vis.size == 0:
        return g2d, pr_s, 0
    inner = {k: tile_box(pr_s["rect"][k], cam, 0) for k in vis}
    outer = {k: tile_box(pr_s["rect"][k], cam, 1) for k in vis}
    boxes = [(b[0] * TILE, b[1] * TILE, b[2] * TILE, b[3] * TILE) for b in outer.values()]
    cand = reach_superset(P, cam, boxes, also=sample[vis])
    pr = oracle.project(P[:, cand], cam)
    # per-tile lists of the tiles any outer box covers, in (fp32 depth bits, index) order
    tiles = set()
    for (x0, y0, x1, y1) in outer.values():
        for ty in range(y0, y1):
            for tx in range(x0, x1):
                tiles.add(ty * cam.tiles_x + tx)
    live = np.nonzero(pr["radius"] > 0)[0]
    rect = pr["rect"][live]
    zb = pr["uvzo"][live, 2].astype(np.float32).view(np.uint32)
    lists = {}
    for (x0, y0, x1, y1) in outer.values():  # members of a box first, then of its tiles
        inbox = np.nonzero((rect[:, 0] < x1) & (rect[:, 2] > x0) & (rect[:, 1] < y1) & (rect[:, 3] > y0))[0]
        rb = rect[inbox]
        for ty in range(y0, y1):
            for tx in range(x0, x1):
                t = ty * cam.tiles_x + tx
                if t in lists:
                    continue
                sel = inbox[(rb[:, 0] <= tx) & (tx < rb[:, 2]) & (rb[:, 1] <= ty) & (ty < rb[:, 3])]
                sel = sel[np.lexsort((cand[live[sel]], zb[sel]))]
                lists[t] = live[sel]
    ranges = np.zeros((cam.tiles_x * cam.tiles_y, 2), np.uint32)
    vals = []
    off = 0
    for t in sorted(tiles):
        vals.append(lists[t].astype(np.uint32))
        ranges[t] = (off, off + len(lists[t]))
        off += len(lists[t])
    vals = np.concatenate(vals) if vals else np.zeros(0, np.uint32)
    img, _, _, _ = oracle.render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, W, H)
    dimg = np.zeros_like(img)
    for k in vis:
        x0, y0, x1, y1 = (v * TILE for v in outer[k])
        x1, y1 = min(x1, W), min(y1, H)
        crop = (slice(None), slice(y0, y1), slice(x0, x1))
        scale = (1.0 / batch) * ((x1 - x0) * (y1 - y0)) / (W * H)
        _, d = oracle.loss(img[crop], target[crop], scale=scale)
        ix0, iy0, ix1, iy1 = (v * TILE for v in inner[k])
        ix1, iy1 = min(ix1, W), min(iy1, H)
        dimg[:, iy0:iy1, ix0:ix1] = d[:, iy0 - y0:iy1 - y0, ix0 - x0:ix1 - x0]
    full = oracle.render_bwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, W, H, dimg)
    pos = np.searchsorted(cand, sample[vis])
    g2d[vis] = full[pos]
    return g2d, pr_s, len(cand)


def sampled_step(P, cams, targets, sample, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-15, step=1):
    """Per-view screen-space gradients, summed parameter gradients and the batch-scaled Adam
    update (t = step, zero moments) of the sampled Gaussians over one batch of views.
    Returns dict(g2d [B, s, 9], grads [15, s, 4], params [15, s, 4], visible [B, s], margin
    [B, s], candidates [B])."""
    B = len(cams)
    s = len(sample)
    out = dict(g2d=np.zeros((B, s, 9)), grads=np.zeros((15, s, 4)), visible=np.zeros((B, s), bool),
               margin=np.zeros((B, s)), candidates=np.zeros(B, np.int64))
    Ps = P[:, sample]
    for b, cam in enumerate(cams):
        g2d, pr_s, nc = view_gradients(P, cam, targets[b], B, sample)
        out["g2d"][b] = g2d
        out["visible"][b] = pr_s["radius"] > 0
        out["margin"][b] = pr_s["margin"]
        out["candidates"][b] = nc
        out["grads"] += oracle.project_bwd(Ps, cam, g2d)
    union = np.nonzero(out["visible"].any(axis=0))[0].astype(np.uint32)
    p, _, _, _ = oracle.sparse_adam(Ps, out["grads"], np.zeros_like(Ps, dtype=np.float64),
                                    np.zeros_like(Ps, dtype=np.float64), union, lr, beta1, beta2, eps, B, step)
    out["params"] = p
    return out


def pick_sample(P, cam, count, seed, rmax, pool=20000):
    """`count` Gaussians visible in this view with radius in [2, rmax] and every projection
    decision well clear of its threshold, chosen by the oracle from a seeded pool."""
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(P.shape[1], min(pool, P.shape[1]), replace=False))
    pr = oracle.project(P[:, idx], cam)
    ok = (pr["radius"] >= 2) & (pr["radius"] <= rmax) & (pr["margin"] >= 1e-4)
    ok &= (np.abs(pr["raw"]) > 1e-3).all(axis=1)  # colour clear of its clamp at 0
    good = idx[ok]
    return np.sort(rng.choice(good, min(count, good.size), replace=False))

