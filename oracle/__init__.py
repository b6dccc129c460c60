"""Python wrapper of the CPU oracle (oracle.cpp) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It compiles ``oracle.cpp`` with g++ (no fast
math, no FMA contraction) into ``liboracle.so`` beside it and calls it through
ctypes.  All arithmetic is in double precision; inputs are converted with
``np.float64`` (exact for float32 data).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
# a test may point the wrapper at another build of the oracle (its mutation checks compile
# deliberately broken copies of oracle.cpp elsewhere and expect the pins to fail on them)
_OVERRIDE = os.environ.get("GS_ORACLE_LIB")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so if missing or older than its source."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                            "-shared", "-o", tmp, _SRC], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        if _OVERRIDE:
            L = C.CDLL(_OVERRIDE)
        else:
            build()
            L = C.CDLL(_LIB)
        dp = C.POINTER(C.c_double)
        ip = C.POINTER(C.c_int32)
        up = C.POINTER(C.c_uint32)
        u64p = C.POINTER(C.c_uint64)
        i64p = C.POINTER(C.c_int64)
        fp = C.POINTER(C.c_float)
        i64, i32, dbl = C.c_int64, C.c_int, C.c_double
        L.oracle_project.argtypes = [dp, i64, dp, i32, i32, dp, dp, ip, dp, ip, ip, dp, dp, dp]
        L.oracle_project.restype = None
        L.oracle_bin_sort.argtypes = [dp, ip, i64, i32, i32, u64p, up, i64, up]
        L.oracle_bin_sort.restype = i64
        L.oracle_render_fwd.argtypes = [dp, dp, dp, up, up, i32, i32, dp, dp, dp, up, dp]
        L.oracle_render_fwd.restype = None
        L.oracle_render_counts.argtypes = [dp, dp, dp, up, up, i32, i32, up, up]
        L.oracle_render_counts.restype = None
        L.oracle_render_bwd.argtypes = [dp, dp, dp, up, up, i32, i32, dp, dp, dp]
        L.oracle_render_bwd.restype = None
        L.oracle_loss.argtypes = [dp, dp, i32, i32, dbl, dbl, dbl, dp]
        L.oracle_loss.restype = dbl
        L.oracle_project_bwd.argtypes = [dp, i64, dp, i32, i32, dp, dp]
        L.oracle_project_bwd.restype = None
        L.oracle_sparse_adam.argtypes = [dp, dp, dp, dp, i64, up, i64, dbl, dbl, dbl, dbl, i32, i64]
        L.oracle_sparse_adam.restype = None
        L.oracle_visible_sets.argtypes = [ip, i32, i64, i64p, up, up, i64p, i64p, fp]
        L.oracle_visible_sets.restype = None
        L.oracle_step.argtypes = [dp, dp, dp, i64, dp, i32, i32, i32, dp, dp, dbl, dbl, dbl, dbl, dbl, dbl,
                                  i64, i32, dp, dp]
        L.oracle_step.restype = dbl
        L.oracle_sh_basis.argtypes = [dp, dp, dp]
        L.oracle_sh_basis.restype = None
        L.oracle_tile_split.argtypes = [up, i32, i32, i32, u64p, u64p, i64p]
        L.oracle_tile_split.restype = None
        L.oracle_view_order.argtypes = [fp, i32, i32, ip, fp]
        L.oracle_view_order.restype = None
        L.oracle_prune.argtypes = [C.c_void_p, i32, i64, C.c_float, C.c_void_p, i64]
        L.oracle_prune.restype = i64
        L.oracle_densify_stat.argtypes = [dp, ip, i64, dp]
        L.oracle_densify_stat.restype = None
        L.oracle_densify.argtypes = [fp, fp, fp, fp, i64, C.c_float, C.c_float, fp, dp, dp, dp, i64, i64p, i64p]
        L.oracle_densify.restype = i64
        _lib = L
    return _lib


def _p(a, t):
    return a.ctypes.data_as(C.POINTER(t)) if a is not None else None


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def cam_array(cam) -> np.ndarray:
    return np.concatenate([np.asarray(cam.R, np.float64).ravel(), np.asarray(cam.t, np.float64),
                           np.array([cam.fx, cam.fy, cam.cx, cam.cy, cam.znear], np.float64)])


def project(params, cam):
    """Projection of every Gaussian.  Returns a dict of arrays (double / int32).  ``margin``:
    relative distance of the nearest decision that can change an output from its threshold
    (culls; the tile rectangle where it would add or drop a tile the Gaussian reaches);
    ``rmargin``: that of the radius ceiling, 0 where the tile rectangle's value may differ
    (the integer outputs radius and tiles)."""
    P = _d(params)
    N = P.shape[1]
    out = dict(uvzo=np.zeros((N, 4)), conic=np.zeros((N, 3)), radius=np.zeros(N, np.int32),
               rgb=np.zeros((N, 3)), rect=np.zeros((N, 4), np.int32), tiles=np.zeros(N, np.int32),
               raw=np.zeros((N, 3)), margin=np.zeros(N), rmargin=np.zeros(N))
    ca = cam_array(cam)
    lib().oracle_project(_p(P, C.c_double), N, _p(ca, C.c_double), cam.width, cam.height,
                         _p(out["uvzo"], C.c_double), _p(out["conic"], C.c_double), _p(out["radius"], C.c_int32),
                         _p(out["rgb"], C.c_double), _p(out["rect"], C.c_int32), _p(out["tiles"], C.c_int32),
                         _p(out["raw"], C.c_double), _p(out["margin"], C.c_double), _p(out["rmargin"], C.c_double))
    return out


def bin_sort(uvzo, radius, width, height):
    """Keys, values and tile ranges of one view (M = len(keys))."""
    U = _d(uvzo)
    R = np.ascontiguousarray(radius, np.int32)
    N = R.shape[0]
    tx, ty = (width + 15) // 16, (height + 15) // 16
    ranges = np.zeros((tx * ty, 2), np.uint32)
    M = lib().oracle_bin_sort(_p(U, C.c_double), _p(R, C.c_int32), N, width, height, None,
                              _p(np.zeros(1, np.uint32), C.c_uint32), 0, _p(ranges, C.c_uint32))
    keys = np.zeros(max(M, 1), np.uint64)
    vals = np.zeros(max(M, 1), np.uint32)
    lib().oracle_bin_sort(_p(U, C.c_double), _p(R, C.c_int32), N, width, height, _p(keys, C.c_uint64),
                          _p(vals, C.c_uint32), M, _p(ranges, C.c_uint32))
    return keys[:M], vals[:M], ranges


def render_fwd(uvzo, conic, rgb, vals, ranges, width, height, bg=(0.0, 0.0, 0.0)):
    P = width * height
    img = np.zeros((3, height, width))
    T = np.zeros((height, width))
    nc = np.zeros((height, width), np.uint32)
    mg = np.zeros((height, width))
    U, Q, Cc, B = _d(uvzo), _d(conic), _d(rgb), _d(bg)
    V = np.ascontiguousarray(vals, np.uint32)
    Rg = np.ascontiguousarray(ranges, np.uint32)
    if V.size == 0:
        V = np.zeros(1, np.uint32)
    lib().oracle_render_fwd(_p(U, C.c_double), _p(Q, C.c_double), _p(Cc, C.c_double), _p(V, C.c_uint32),
                            _p(Rg, C.c_uint32), width, height, _p(B, C.c_double), _p(img, C.c_double),
                            _p(T, C.c_double), _p(nc, C.c_uint32), _p(mg, C.c_double))
    del P
    return img, T, nc, mg


def render_counts(uvzo, conic, rgb, vals, ranges, width, height):
    """Per-pixel work of the compositing walk, two [H][W] uint32 arrays: entries evaluated
    (through the one that would take the transmittance below 1e-4, else the whole tile list)
    and entries accumulated."""
    U, Q, Cc = _d(uvzo), _d(conic), _d(rgb)
    V = np.ascontiguousarray(vals, np.uint32)
    if V.size == 0:
        V = np.zeros(1, np.uint32)
    Rg = np.ascontiguousarray(ranges, np.uint32)
    n_eval = np.zeros((height, width), np.uint32)
    n_used = np.zeros((height, width), np.uint32)
    lib().oracle_render_counts(_p(U, C.c_double), _p(Q, C.c_double), _p(Cc, C.c_double), _p(V, C.c_uint32),
                               _p(Rg, C.c_uint32), width, height, _p(n_eval, C.c_uint32), _p(n_used, C.c_uint32))
    return n_eval, n_used


def render_bwd(uvzo, conic, rgb, vals, ranges, width, height, dimg, bg=(0.0, 0.0, 0.0)):
    """Per-Gaussian screen-space gradients, N x 9: du, dv, dA, dB, dC, dopacity, dr, dg, db."""
    U, Q, Cc, B, D = _d(uvzo), _d(conic), _d(rgb), _d(bg), _d(dimg)
    N = U.shape[0]
    g2d = np.zeros((N, 9))
    V = np.ascontiguousarray(vals, np.uint32)
    if V.size == 0:
        V = np.zeros(1, np.uint32)
    Rg = np.ascontiguousarray(ranges, np.uint32)
    lib().oracle_render_bwd(_p(U, C.c_double), _p(Q, C.c_double), _p(Cc, C.c_double), _p(V, C.c_uint32),
                            _p(Rg, C.c_uint32), width, height, _p(B, C.c_double), _p(D, C.c_double),
                            _p(g2d, C.c_double))
    return g2d


def loss(img, target, w_l1=0.8, w_ssim=0.2, scale=1.0, grad=True):
    X, Y = _d(img), _d(target)
    H, W = X.shape[1], X.shape[2]
    d = np.zeros_like(X) if grad else None
    val = lib().oracle_loss(_p(X, C.c_double), _p(Y, C.c_double), W, H, w_l1, w_ssim, scale,
                            _p(d, C.c_double))
    return val, d


def project_bwd(params, cam, g2d):
    P = _d(params)
    N = P.shape[1]
    G = _d(g2d)
    grads = np.zeros_like(P)
    ca = cam_array(cam)
    lib().oracle_project_bwd(_p(P, C.c_double), N, _p(ca, C.c_double), cam.width, cam.height, _p(G, C.c_double),
                             _p(grads, C.c_double))
    return grads


def sparse_adam(params, grads, m, v, idx, lr, beta1, beta2, eps, batch, step):
    """Returns updated (params, grads, m, v) as new double arrays."""
    P, G, Mm, Vv = _d(params).copy(), _d(grads).copy(), _d(m).copy(), _d(v).copy()
    N = P.shape[1]
    I = np.ascontiguousarray(idx, np.uint32)
    if I.size == 0:
        I = np.zeros(1, np.uint32)
        n_idx = 0
    else:
        n_idx = len(idx)
    lib().oracle_sparse_adam(_p(P, C.c_double), _p(G, C.c_double), _p(Mm, C.c_double), _p(Vv, C.c_double), N,
                             _p(I, C.c_uint32), n_idx, lr, beta1, beta2, eps, batch, step)
    return P, G, Mm, Vv


def visible_sets(radii):
    """radii: B x N int32.  Returns offsets, indices, union, inter (B x B), jaccard (B x B)."""
    R = np.ascontiguousarray(radii, np.int32)
    B, N = R.shape
    tot = int((R > 0).sum())
    off = np.zeros(B + 1, np.int64)
    ind = np.zeros(max(tot, 1), np.uint32)
    uni = np.zeros(max(N, 1), np.uint32)
    nu = np.zeros(1, np.int64)
    inter = np.zeros((B, B), np.int64)
    jac = np.zeros((B, B), np.float32)
    lib().oracle_visible_sets(_p(R, C.c_int32), B, N, _p(off, C.c_int64), _p(ind, C.c_uint32), _p(uni, C.c_uint32),
                              _p(nu, C.c_int64), _p(inter, C.c_int64), _p(jac, C.c_float))
    return off, ind[:tot], uni[: int(nu[0])], inter, jac


def tile_split(cost_px, parts):
    """cost_px: H x W uint32 per-pixel costs.  Returns (tile_cost [T] uint64, cum [T] uint64,
    bounds [parts + 1] int64): block k of the split holds tiles [bounds[k], bounds[k + 1])."""
    c = np.ascontiguousarray(cost_px, np.uint32)
    H, W = c.shape
    T = ((W + 15) // 16) * ((H + 15) // 16)
    tc = np.zeros(T, np.uint64)
    cum = np.zeros(T, np.uint64)
    bounds = np.zeros(parts + 1, np.int64)
    lib().oracle_tile_split(_p(c, C.c_uint32), W, H, parts, _p(tc, C.c_uint64), _p(cum, C.c_uint64),
                            _p(bounds, C.c_int64))
    return tc, cum, bounds


def view_order(weights, unit=1):
    """weights: B x B float32 (the Jaccard matrix).  Returns (order [B] int32, score [B] float32)."""
    w = np.ascontiguousarray(weights, np.float32)
    B = w.shape[0]
    order = np.zeros(B, np.int32)
    score = np.zeros(B, np.float32)
    lib().oracle_view_order(_p(w, C.c_float), B, unit, _p(order, C.c_int32), _p(score, C.c_float))
    return order, score


def prune(plane_sets, min_logit):
    """plane_sets: list of float32 [15, N, 4] arrays (parameters first: its plane 0, w is the
    opacity logit).  Returns (kept count, list of [15, kept, 4] arrays)."""
    sets = [np.ascontiguousarray(p, np.float32) for p in plane_sets]
    n = sets[0].shape[1]
    outs = [np.zeros((15, max(n, 1), 4), np.float32) for _ in sets]
    ins = (C.c_void_p * len(sets))(*[p.ctypes.data for p in sets])
    ous = (C.c_void_p * len(sets))(*[o.ctypes.data for o in outs])
    k = lib().oracle_prune(C.cast(ins, C.c_void_p), len(sets), n, C.c_float(min_logit), C.cast(ous, C.c_void_p),
                           max(n, 1))
    # the kernel layout keeps the plane stride; re-pack to a stride of k
    return k, [np.ascontiguousarray(o[:, :k]) for o in outs]


def densify_stat(g2d, radius, stat=None):
    """Adds one view's densification statistic: for radius > 0, |(du, dv)| and one view.
    g2d: N x 9 (oracle layout); returns the N x 2 statistic (a new array unless given)."""
    G = _d(g2d)
    R = np.ascontiguousarray(radius, np.int32)
    N = R.shape[0]
    out = np.zeros((N, 2)) if stat is None else np.ascontiguousarray(stat, np.float64)
    lib().oracle_densify_stat(_p(G, C.c_double), _p(R, C.c_int32), N, _p(out, C.c_double))
    return out


def densify(params, m, v, stat, grad_threshold, log_scale_threshold, normals):
    """Clone / split.  params, m, v: float32 [15, N, 4]; stat: float32 N x 2 (sum of screen
    gradient lengths, views); normals: float32 N x 6.  Returns (params, m, v) as double
    [15, n_out, 4] arrays and (n_clone, n_split)."""
    P, Mm, Vv = (np.ascontiguousarray(a, np.float32) for a in (params, m, v))
    S = np.ascontiguousarray(stat, np.float32)
    Z = np.ascontiguousarray(normals, np.float32)
    N = P.shape[1]
    nc, ns = np.zeros(1, np.int64), np.zeros(1, np.int64)
    args = lambda op, om, ov, stride: (_p(P, C.c_float), _p(Mm, C.c_float), _p(Vv, C.c_float), _p(S, C.c_float), N,
                                       C.c_float(grad_threshold), C.c_float(log_scale_threshold), _p(Z, C.c_float),
                                       _p(op, C.c_double), _p(om, C.c_double), _p(ov, C.c_double), stride,
                                       _p(nc, C.c_int64), _p(ns, C.c_int64))
    dummy = np.zeros(1)
    n_out = lib().oracle_densify(*args(dummy, dummy, dummy, 0))
    outs = [np.zeros((15, max(n_out, 1), 4)) for _ in range(3)]
    lib().oracle_densify(*args(outs[0], outs[1], outs[2], n_out))
    return tuple(o[:, :n_out] for o in outs), (int(nc[0]), int(ns[0]))


def step(params, m, v, cams, targets, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-15, t=1, w_l1=0.8, w_ssim=0.2,
         bg=(0.0, 0.0, 0.0), do_adam=True):
    """One training step over the views ``cams`` (all the same size).

    Returns dict(loss, grads, params, m, v, images) in double precision.
    """
    P, Mm, Vv = _d(params).copy(), _d(m).copy(), _d(v).copy()
    N = P.shape[1]
    B = len(cams)
    W, H = cams[0].width, cams[0].height
    ca = np.concatenate([cam_array(c) for c in cams])
    T = _d(targets)
    Bg = _d(bg)
    grads = np.zeros_like(P)
    imgs = np.zeros((B, 3, H, W))
    val = lib().oracle_step(_p(P, C.c_double), _p(Mm, C.c_double), _p(Vv, C.c_double), N, _p(ca, C.c_double), B, W,
                            H, _p(T, C.c_double), _p(Bg, C.c_double), w_l1, w_ssim, lr, beta1, beta2, eps, t,
                            1 if do_adam else 0, _p(grads, C.c_double), _p(imgs, C.c_double))
    return dict(loss=val, grads=grads, params=P, m=Mm, v=Vv, images=imgs)


def sh_basis(d):
    D = _d(d)
    Y = np.zeros(16)
    dY = np.zeros(48)
    lib().oracle_sh_basis(_p(D, C.c_double), _p(Y, C.c_double), _p(dY, C.c_double))
    return Y, dY.reshape(16, 3)


def render_view(params, cam, bg=(0.0, 0.0, 0.0)):
    """Forward render of one view through the oracle stages (project, bin, composite)."""
    pr = project(params, cam)
    keys, vals, ranges = bin_sort(pr["uvzo"], pr["radius"], cam.width, cam.height)
    img, T, nc, mg = render_fwd(pr["uvzo"], pr["conic"], pr["rgb"], vals, ranges, cam.width, cam.height, bg)
    return img
