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


def max_scale_sq(P):
    """s_max^2 of every Gaussian (view-independent: computed once per scene)."""
    return np.exp(2.0 * P[1, :, :3].max(axis=1)).astype(np.float32)


def reach_superset(P, cam, tile_mask, also=(), s2max=None):
    """Indices of every Gaussian whose tile rectangle can meet a tile marked in tile_mask
    [Ty, Tx] in this view.  The projected radius obeys
    r = ceil(3 sqrt(lambda_max)) <= 3 sqrt((f/z)^2 (2 + xr^2 + yr^2) s_max^2 + 0.3) + 1
    (the Frobenius norm of the Jacobian bounds its spectral norm; xr, yr are the clamped
    ratios), and the rectangle spans [floor(u) - r, floor(u) + r] rounded out to tiles, so it
    stays within r + 17 pixels of (u, v); the marked tiles in that reach are counted with a
    2-D prefix sum of the mask."""
    R = np.asarray(cam.R, np.float32)
    t = np.asarray(cam.t, np.float32)
    Ty, Tx = tile_mask.shape
    S = np.zeros((Ty + 1, Tx + 1), np.int64)
    S[1:, 1:] = tile_mask.astype(np.int64).cumsum(0).cumsum(1)
    n = P.shape[1]
    keep = np.zeros(n, bool)
    limx = np.float32(1.3 * (cam.width / 2.0) / cam.fx)
    limy = np.float32(1.3 * (cam.height / 2.0) / cam.fy)
    f = np.float32(max(cam.fx, cam.fy))
    if s2max is None:
        s2max = max_scale_sq(P)
    step = 4_000_000
    for a in range(0, n, step):
        # float32 is enough for a bound with pixels of slack: the reach gets 4 more pixels
        pc = P[0, a:a + step, :3] @ R.T
        pc += t
        z = pc[:, 2]
        front = z > np.float32(0.99 * cam.znear)
        iz = np.float32(1.0) / np.where(front, z, np.float32(1.0))
        x = pc[:, 0] * iz
        y = pc[:, 1] * iz
        lam = np.square(np.clip(x, -limx, limx))
        lam += np.square(np.clip(y, -limy, limy))
        lam += np.float32(2.0)
        lam *= np.square(f * iz)
        lam *= s2max[a:a + step]
        lam += np.float32(0.3)
        r = np.sqrt(lam)
        r *= np.float32(3.0)
        r += np.float32(1.0 + TILE + 1.0 + 4.0)
        u = x * np.float32(cam.fx) + np.float32(cam.cx)
        v = y * np.float32(cam.fy) + np.float32(cam.cy)
        inside = front & (u + r >= 0) & (u - r <= cam.width) & (v + r >= 0) & (v - r <= cam.height)
        tx0 = np.clip((u - r) // TILE, 0, Tx - 1).astype(np.int64)
        tx1 = np.clip((u + r) // TILE, 0, Tx - 1).astype(np.int64) + 1
        ty0 = np.clip((v - r) // TILE, 0, Ty - 1).astype(np.int64)
        ty1 = np.clip((v + r) // TILE, 0, Ty - 1).astype(np.int64) + 1
        cnt = S[ty1, tx1] - S[ty0, tx1] - S[ty1, tx0] + S[ty0, tx0]
        keep[a:a + step] = inside & (cnt > 0)
    keep[np.asarray(also, np.int64)] = True
    return np.nonzero(keep)[0]


def project_subset(P, idx, cam, chunk=1_000_000):
    """oracle.project of the Gaussians idx, in chunks (bounds the double-precision copies)."""
    keys = ("uvzo", "conic", "rgb", "radius", "rect")
    parts = {k: [] for k in keys}
    for a in range(0, len(idx), chunk):
        pr = oracle.project(P[:, idx[a:a + chunk]], cam)
        for k in keys:
            parts[k].append(pr[k])
    return {k: np.concatenate(v) for k, v in parts.items()}


def tile_box(rect, cam, grow):
    """Tile rectangle [x0, x1) x [y0, y1) grown by `grow` tiles, clipped to the image."""
    x0, y0, x1, y1 = (int(v) for v in rect)
    return (max(0, x0 - grow), max(0, y0 - grow), min(cam.tiles_x, x1 + grow), min(cam.tiles_y, y1 + grow))


def view_gradients(P, cam, target, batch, sample, s2max=None):
    """Screen-space gradients (n x 9, oracle layout) of the sampled Gaussians in one view, the
    oracle's projection of them (dict), the number of candidate Gaussians looked at, and the
    part of the screen-space gradients that comes from pixels whose compositing decisions sit
    within 1e-5 of a threshold."""
    W, H = cam.width, cam.height
    pr_s = oracle.project(P[:, sample], cam)
    vis = np.nonzero(pr_s["radius"] > 0)[0]
    g2d = np.zeros((len(sample), 9))
    g2d_flag = np.zeros((len(sample), 9))
    if vis.size == 0:
        return g2d, pr_s, 0, g2d_flag
    inner = {k: tile_box(pr_s["rect"][k], cam, 0) for k in vis}
    outer = {k: tile_box(pr_s["rect"][k], cam, 1) for k in vis}
    mask = np.zeros((cam.tiles_y, cam.tiles_x), bool)
    for (x0, y0, x1, y1) in outer.values():
        mask[y0:y1, x0:x1] = True
    cand = reach_superset(P, cam, mask, also=sample[vis], s2max=s2max)
    pr = project_subset(P, cand, cam)
    live = np.nonzero(pr["radius"] > 0)[0]
    rect = pr["rect"][live]
    zb = pr["uvzo"][live, 2].astype(np.float32).view(np.uint32)
    for k in vis:
        # the crop: the outer box on its own tile grid (its origin is a tile corner, so the
        # tiles and pixel centres are those of the whole view, shifted)
        x0, y0, x1, y1 = outer[k]
        cw, ch = min(x1 * TILE, W) - x0 * TILE, min(y1 * TILE, H) - y0 * TILE
        ctx = x1 - x0
        inbox = np.nonzero((rect[:, 0] < x1) & (rect[:, 2] > x0) & (rect[:, 1] < y1) & (rect[:, 3] > y0))[0]
        rb = rect[inbox]
        ranges = np.zeros(((y1 - y0) * ctx, 2), np.uint32)
        vals, off = [], 0
        for ty in range(y0, y1):
            for tx in range(x0, x1):
                sel = np.nonzero((rb[:, 0] <= tx) & (tx < rb[:, 2]) & (rb[:, 1] <= ty) & (ty < rb[:, 3]))[0]
                sel = sel[np.lexsort((cand[live[inbox[sel]]], zb[inbox[sel]]))]  # (depth bits, index)
                vals.append(sel.astype(np.uint32))
                ranges[(ty - y0) * ctx + (tx - x0)] = (off, off + len(sel))
                off += len(sel)
        vals = np.concatenate(vals)
        g = live[inbox]
        uvzo = pr["uvzo"][g].copy()
        uvzo[:, 0] -= x0 * TILE
        uvzo[:, 1] -= y0 * TILE
        conic, rgb = pr["conic"][g], pr["rgb"][g]
        img, _, _, mg = oracle.render_fwd(uvzo, conic, rgb, vals, ranges, cw, ch)
        crop = (slice(None), slice(y0 * TILE, y0 * TILE + ch), slice(x0 * TILE, x0 * TILE + cw))
        scale = (1.0 / batch) * (cw * ch) / (W * H)
        _, d = oracle.loss(img, target[crop], scale=scale)
        keep = np.zeros_like(d)
        ix0, iy0, ix1, iy1 = inner[k]
        sl = (slice(None), slice((iy0 - y0) * TILE, min(iy1 * TILE, H) - y0 * TILE),
              slice((ix0 - x0) * TILE, min(ix1 * TILE, W) - x0 * TILE))
        keep[sl] = d[sl]
        full = oracle.render_bwd(uvzo, conic, rgb, vals, ranges, cw, ch, keep)
        pos = np.nonzero(cand[g] == sample[k])[0]
        assert pos.size == 1
        g2d[k] = full[pos[0]]
        flagged = mg < 1e-5
        if flagged.any():
            part = oracle.render_bwd(uvzo, conic, rgb, vals, ranges, cw, ch, keep * flagged[None])
            g2d_flag[k] = part[pos[0]]
    return g2d, pr_s, len(cand), g2d_flag


_SHARED = {}


def _attach(name, shape, s2name):
    from multiprocessing import shared_memory

    shm = shared_memory.SharedMemory(name=name)
    sh2 = shared_memory.SharedMemory(name=s2name)
    _SHARED["P"] = np.ndarray(shape, np.float32, buffer=shm.buf)
    _SHARED["s2"] = np.ndarray((shape[1],), np.float32, buffer=sh2.buf)
    _SHARED["keep"] = (shm, sh2)


def _view_job(args):
    cam, target, batch, sample = args
    g2d, pr_s, nc, g2f = view_gradients(_SHARED["P"], cam, target, batch, sample, _SHARED["s2"])
    return g2d, pr_s["radius"], pr_s["margin"], nc, g2f


def _per_view(P, cams, targets, sample, workers):
    """view_gradients of every view: in this process, or in `workers` spawned processes that
    share the parameters through shared memory."""
    B = len(cams)
    s2 = max_scale_sq(P)
    if workers <= 1 or B == 1:
        res = []
        for b, cam in enumerate(cams):
            g2d, pr_s, nc, g2f = view_gradients(P, cam, targets[b], B, sample, s2)
            res.append((g2d, pr_s["radius"], pr_s["margin"], nc, g2f))
        return res
    import multiprocessing as mp
    from multiprocessing import shared_memory

    try:
        shm = shared_memory.SharedMemory(create=True, size=P.nbytes)
        sh2 = shared_memory.SharedMemory(create=True, size=s2.nbytes)
    except OSError:  # no room for a shared copy: one view after another in this process
        return _per_view(P, cams, targets, sample, 1)
    try:
        np.ndarray(P.shape, np.float32, buffer=shm.buf)[...] = P
        np.ndarray(s2.shape, np.float32, buffer=sh2.buf)[...] = s2
        ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
        with ctx.Pool(min(workers, B), initializer=_attach, initargs=(shm.name, P.shape, sh2.name)) as pool:
            res = pool.map(_view_job, [(cam, targets[b], B, sample) for b, cam in enumerate(cams)])
    finally:
        shm.close()
        shm.unlink()
        sh2.close()
        sh2.unlink()
    return res


def sampled_step(P, cams, targets, sample, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-15, step=1, workers=1):
    """Per-view screen-space gradients, summed parameter gradients and the batch-scaled Adam
    update (t = step, zero moments) of the sampled Gaussians over one batch of views.
    Returns dict(g2d [B, s, 9], grads [15, s, 4], params [15, s, 4], visible [B, s], margin
    [B, s], candidates [B], g2d_flag [B, s, 9], grads_flag [15, s, 4]: the parts of the
    gradients that come from pixels with a compositing decision on its threshold)."""
    B = len(cams)
    s = len(sample)
    out = dict(g2d=np.zeros((B, s, 9)), grads=np.zeros((15, s, 4)), visible=np.zeros((B, s), bool),
               margin=np.zeros((B, s)), candidates=np.zeros(B, np.int64), g2d_flag=np.zeros((B, s, 9)),
               grads_flag=np.zeros((15, s, 4)))
    Ps = P[:, sample]
    per_view = _per_view(np.ascontiguousarray(P, np.float32), cams, targets, sample, workers)
    for b, cam in enumerate(cams):
        g2d, radius, margin, nc, g2f = per_view[b]
        out["g2d_flag"][b] = g2f
        out["grads_flag"] += oracle.project_bwd(Ps, cam, g2f)
        out["g2d"][b] = g2d
        out["visible"][b] = radius > 0
        out["margin"][b] = margin
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

