"""ctypes binding of libgs.so: one Python function per C entry point, argument marshalling only.

Arguments that are device arrays accept a torch CUDA tensor or an integer device address.
``stream`` accepts a ``torch.cuda.Stream``, an integer ``cudaStream_t`` or None (the current
torch stream).  A nonzero status raises ``GSError`` carrying ``gs_last_error()``.  The
library must have been built (``gaussian_splatting_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgs.so")

GS_OK, GS_ERR_INVALID, GS_ERR_CUDA, GS_ERR_CAPACITY, GS_ERR_TIMEOUT = 0, 1, 2, 3, 4
_NAMES = {1: "GS_ERR_INVALID", 2: "GS_ERR_CUDA", 3: "GS_ERR_CAPACITY", 4: "GS_ERR_TIMEOUT"}

# every symbol include/gs.h declares
EXPORTS = ["gs_last_error", "gs_version", "gs_project", "gs_project_batch", "gs_bin_sort_workspace_size", "gs_bin_sort",
           "gs_bin_sort_batch_workspace_size", "gs_bin_sort_batch",
           "gs_render_fwd", "gs_tile_order", "gs_loss_workspace_size", "gs_loss", "gs_loss_noalloc", "gs_render_bwd", "gs_project_bwd",
           "gs_visible_sets_workspace_size", "gs_visible_sets", "gs_sparse_adam", "gs_project_bwd_adam",
           "gs_tile_split", "gs_view_order", "gs_prune_workspace_size", "gs_prune", "gs_densify_workspace_size",
           "gs_densify", "gs_probe_ffma",
           "gs_debug_set_wait_limit",
           "gs_debug_drop_publish"]


class GSError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: {_NAMES.get(status, status)}: {msg}")
        self.status = status


class Camera(C.Structure):
    _fields_ = [("R", C.c_float * 9), ("t", C.c_float * 3), ("fx", C.c_float), ("fy", C.c_float),
                ("cx", C.c_float), ("cy", C.c_float), ("znear", C.c_float), ("width", C.c_int32),
                ("height", C.c_int32)]


def camera(cam) -> Camera:
    """gs_camera from any object with R, t, fx, fy, cx, cy, znear, width, height."""
    c = Camera()
    R = [float(x) for x in np.asarray(cam.R, dtype=np.float32).ravel()]
    t = [float(x) for x in np.asarray(cam.t, dtype=np.float32).ravel()]
    c.R[:] = R
    c.t[:] = t
    c.fx, c.fy, c.cx, c.cy, c.znear = cam.fx, cam.fy, cam.cx, cam.cy, cam.znear
    c.width, c.height = cam.width, cam.height
    return c


_lib = None


def load() -> C.CDLL:
    """Load libgs.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libgs.so not built at {LIB_PATH}; run `python -m gaussian_splatting_gb300.build`")
    L = C.CDLL(LIB_PATH)
    vp, i64, i32, f32, sz = C.c_void_p, C.c_int64, C.c_int, C.c_float, C.c_size_t
    cp = C.POINTER(Camera)
    sig = {
        "gs_last_error": ([], C.c_char_p),
        "gs_version": ([], C.c_int),
        "gs_project": ([vp, i64, cp, vp, vp], i32),
        "gs_project_batch": ([vp, i64, vp, i32, vp, vp, i64, vp], i32),
        "gs_bin_sort_workspace_size": ([i64, i64, cp], sz),
        "gs_bin_sort": ([vp, i64, cp, vp, sz, vp, vp, i64, vp, vp, vp, vp], i32),
        "gs_bin_sort_batch_workspace_size": ([i32, i64, i64, vp], sz),
        "gs_bin_sort_batch": ([vp, i32, i64, vp, vp, sz, vp, vp, i64, vp, vp, vp, vp], i32),
        "gs_render_fwd": ([vp, i64, vp, vp, cp, vp, vp, vp, vp, vp, vp, vp, vp], i32),
        "gs_tile_order": ([vp, vp, i32, i32, i32, vp, vp], i32),
        "gs_loss_workspace_size": ([i32, i32], sz),
        "gs_loss": ([vp, vp, i32, i32, f32, f32, f32, vp, i32, vp, vp, sz, vp], i32),
        "gs_loss_noalloc": ([vp, vp, i32, i32, f32, f32, f32, vp, i32, vp, vp], i32),
        "gs_render_bwd": ([vp, i64, vp, vp, cp, vp, vp, vp, vp, vp, vp, vp], i32),
        "gs_project_bwd": ([vp, i64, cp, vp, vp, vp, vp, vp], i32),
        "gs_visible_sets_workspace_size": ([i32, i64], sz),
        "gs_visible_sets": ([vp, i32, i64, vp, sz, vp, vp, vp, vp, vp, vp, vp, i64, vp], i32),
        "gs_sparse_adam": ([vp, vp, vp, vp, i64, vp, vp, i64, f32, f32, f32, f32, i32, i64, vp, i32, vp], i32),
        "gs_project_bwd_adam": ([vp, i64, vp, i32, vp, vp, vp, vp, f32, f32, f32, f32, i64, vp, i32, vp, vp, i64, vp],
                                i32),
        "gs_tile_split": ([vp, i32, i32, i32, vp, vp, vp, vp], i32),
        "gs_view_order": ([vp, i32, i32, vp, vp, vp], i32),
        "gs_prune_workspace_size": ([i64], sz),
        "gs_prune": ([vp, i32, i64, f32, vp, i64, vp, sz, vp, vp, vp], i32),
        "gs_densify_workspace_size": ([i64], sz),
        "gs_densify": ([vp, vp, vp, i64, vp, f32, f32, vp, vp, vp, vp, i64, vp, sz, vp, vp, vp], i32),
        "gs_probe_ffma": ([vp, i32, i32, vp], i32),
        "gs_debug_set_wait_limit": ([i64], None),
        "gs_debug_drop_publish": ([i32], None),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, where: str):
    if status != GS_OK:
        raise GSError(status, where, load().gs_last_error().decode())


def _cam(cam):
    return C.byref(cam if isinstance(cam, Camera) else camera(cam))


def _floats3(bg):
    if bg is None:
        return None
    arr = (C.c_float * 3)(*[float(x) for x in bg])
    return C.cast(arr, C.c_void_p), arr


def version() -> int:
    return load().gs_version()


def gs_project(params, n, cam, proj, stream=None):
    _check(load().gs_project(_ptr(params), n, _cam(cam), _ptr(proj), _stream(stream)), "gs_project")


def gs_project_batch(params, n, cams, projs, stream=None, visible_bits=None, bits_stride=0):
    """gs_project for len(cams) views; projs is a list of per-view [3][n][4] outputs;
    visible_bits (optional) receives the views' visibility bitsets."""
    c, p = _cams(cams), _ptrs(projs)
    _check(load().gs_project_batch(_ptr(params), n, c[0], len(cams), p[0], _ptr(visible_bits),
                                   bits_stride if visible_bits is not None else 0, _stream(stream)),
           "gs_project_batch")


def gs_bin_sort_workspace_size(n, capacity, cam) -> int:
    return load().gs_bin_sort_workspace_size(n, capacity, _cam(cam))


def gs_bin_sort(proj, n, cam, workspace, workspace_bytes, keys, vals, capacity, ranges, count, sync=False,
                stream=None):
    """Returns M (host int) when sync=True, else None (M stays in count[0] on the device)."""
    host = C.c_int64(0)
    _check(load().gs_bin_sort(_ptr(proj), n, _cam(cam), _ptr(workspace), workspace_bytes, _ptr(keys), _ptr(vals),
                              capacity, _ptr(ranges), _ptr(count), C.byref(host) if sync else None,
                              _stream(stream)), "gs_bin_sort")
    return host.value if sync else None


def _cams(cams):
    arr = (Camera * len(cams))(*[c if isinstance(c, Camera) else camera(c) for c in cams])
    return C.cast(arr, C.c_void_p), arr


def _ptrs(xs):
    arr = (C.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    return C.cast(arr, C.c_void_p), arr


def gs_bin_sort_batch_workspace_size(batch, n, capacity, cams) -> int:
    c = _cams(cams[:batch])
    return load().gs_bin_sort_batch_workspace_size(batch, n, capacity, c[0])


def gs_bin_sort_batch(projs, n, cams, workspace, workspace_bytes, keys, vals, capacity, ranges, counts, sync=False,
                      stream=None):
    """gs_bin_sort for len(cams) views; keys may be None or a list with None entries.  Returns
    the per-view M (host list) when sync=True, else None."""
    batch = len(cams)
    c, p, v, r = _cams(cams), _ptrs(projs), _ptrs(vals), _ptrs(ranges)
    k = _ptrs(keys) if keys is not None else (None, None)
    host = (C.c_int64 * batch)()
    _check(load().gs_bin_sort_batch(p[0], batch, n, c[0], _ptr(workspace), workspace_bytes, k[0], v[0], capacity,
                                    r[0], _ptr(counts), C.cast(host, C.c_void_p) if sync else None,
                                    _stream(stream)), "gs_bin_sort_batch")
    return list(host) if sync else None


def gs_render_fwd(proj, n, vals, ranges, cam, bg, image, T_final, n_contrib, work=None, stream=None,
                  tile_order=None, tile_cost=None):
    b = _floats3(bg)
    _check(load().gs_render_fwd(_ptr(proj), n, _ptr(vals), _ptr(ranges), _cam(cam), b[0] if b else None,
                                _ptr(image), _ptr(T_final), _ptr(n_contrib), _ptr(work), _ptr(tile_order),
                                _ptr(tile_cost), _stream(stream)), "gs_render_fwd")


def gs_tile_order(ranges, tile_cost, tiles_x, tiles_y, order, block=1, stream=None):
    _check(load().gs_tile_order(_ptr(ranges), _ptr(tile_cost), tiles_x, tiles_y, block, _ptr(order),
                                _stream(stream)), "gs_tile_order")


def gs_loss_workspace_size(width, height) -> int:
    return load().gs_loss_workspace_size(width, height)


def gs_loss(image, target, width, height, w_l1, w_ssim, scale, loss_dev, accumulate, dL_dimage, workspace,
            workspace_bytes, stream=None):
    _check(load().gs_loss(_ptr(image), _ptr(target), width, height, w_l1, w_ssim, scale, _ptr(loss_dev),
                          1 if accumulate else 0, _ptr(dL_dimage), _ptr(workspace), workspace_bytes,
                          _stream(stream)), "gs_loss")


def gs_loss_noalloc(image, target, width, height, w_l1, w_ssim, scale, loss_dev, accumulate, dL_dimage,
                    stream=None):
    """gs_loss without a workspace (partial sums in a fixed array inside the library)."""
    _check(load().gs_loss_noalloc(_ptr(image), _ptr(target), width, height, w_l1, w_ssim, scale, _ptr(loss_dev),
                                  1 if accumulate else 0, _ptr(dL_dimage), _stream(stream)), "gs_loss_noalloc")


def gs_render_bwd(proj, n, vals, ranges, cam, bg, T_final, n_contrib, dL_dimage, grad2d, stream=None,
                  tile_order=None):
    b = _floats3(bg)
    _check(load().gs_render_bwd(_ptr(proj), n, _ptr(vals), _ptr(ranges), _cam(cam), b[0] if b else None,
                                _ptr(T_final), _ptr(n_contrib), _ptr(dL_dimage), _ptr(grad2d), _ptr(tile_order),
                                _stream(stream)), "gs_render_bwd")


def gs_project_bwd(params, n, cam, proj, grad2d, grads, densify_stat=None, stream=None):
    _check(load().gs_project_bwd(_ptr(params), n, _cam(cam), _ptr(proj), _ptr(grad2d), _ptr(grads),
                                 _ptr(densify_stat), _stream(stream)), "gs_project_bwd")


def gs_visible_sets_workspace_size(batch, n) -> int:
    return load().gs_visible_sets_workspace_size(batch, n)


def gs_visible_sets(projs, batch, n, workspace, workspace_bytes, offsets, indices, union_idx, n_union, inter,
                    jaccard, stream=None, visible_bits=None, bits_stride=0):
    arr = (C.c_void_p * batch)(*[_ptr(p) for p in projs]) if projs is not None else None
    _check(load().gs_visible_sets(C.cast(arr, C.c_void_p) if arr is not None else None, batch, n, _ptr(workspace),
                                  workspace_bytes, _ptr(offsets), _ptr(indices), _ptr(union_idx), _ptr(n_union),
                                  _ptr(inter), _ptr(jaccard), _ptr(visible_bits),
                                  bits_stride if visible_bits is not None else 0, _stream(stream)), "gs_visible_sets")


def gs_sparse_adam(params, grads, exp_avg, exp_avg_sq, n, idx, n_idx, max_idx, lr, beta1, beta2, eps, batch, step,
                   counts=None, n_counts=0, stream=None):
    _check(load().gs_sparse_adam(_ptr(params), _ptr(grads), _ptr(exp_avg), _ptr(exp_avg_sq), n, _ptr(idx),
                                 _ptr(n_idx), max_idx, lr, beta1, beta2, eps, batch, step, _ptr(counts),
                                 n_counts if counts is not None else 0, _stream(stream)), "gs_sparse_adam")


def gs_project_bwd_adam(params, n, cams, projs, grad2ds, exp_avg, exp_avg_sq, lr, beta1, beta2, eps, step,
                        counts=None, n_counts=0, densify_stat=None, stream=None, visible_bits=None, bits_stride=0):
    batch = len(cams)
    carr = (Camera * batch)(*[c if isinstance(c, Camera) else camera(c) for c in cams])
    parr = (C.c_void_p * batch)(*[_ptr(p) for p in projs])
    garr = (C.c_void_p * batch)(*[_ptr(g) for g in grad2ds])
    _check(load().gs_project_bwd_adam(_ptr(params), n, C.cast(carr, C.c_void_p), batch, C.cast(parr, C.c_void_p),
                                      C.cast(garr, C.c_void_p), _ptr(exp_avg), _ptr(exp_avg_sq), lr, beta1, beta2,
                                      eps, step, _ptr(counts), n_counts if counts is not None else 0,
                                      _ptr(densify_stat), _ptr(visible_bits), bits_stride if visible_bits is not None else 0,
                                      _stream(stream)), "gs_project_bwd_adam")


def gs_tile_split(cost_px, width, height, parts, tile_cost, cum, bounds, stream=None):
    _check(load().gs_tile_split(_ptr(cost_px), width, height, parts, _ptr(tile_cost), _ptr(cum), _ptr(bounds),
                                _stream(stream)), "gs_tile_split")


def gs_view_order(weights, batch, unit, order, score, stream=None):
    _check(load().gs_view_order(_ptr(weights), batch, unit, _ptr(order), _ptr(score), _stream(stream)),
           "gs_view_order")


def gs_prune_workspace_size(n) -> int:
    return load().gs_prune_workspace_size(n)


def gs_prune(planes_in, n, min_logit, planes_out, out_stride, workspace, n_keep, sync=False, stream=None):
    """Returns the kept count (host int) when sync=True, else None (it stays in n_keep)."""
    pin = _ptrs(planes_in)
    pout = _ptrs(planes_out) if planes_out is not None else (None, None)
    host = C.c_int64(0)
    _check(load().gs_prune(pin[0], len(planes_in), n, min_logit, pout[0], out_stride, _ptr(workspace),
                           workspace.numel() if workspace is not None else 0, _ptr(n_keep),
                           C.byref(host) if sync else None, _stream(stream)), "gs_prune")
    return host.value if sync else None


def gs_densify_workspace_size(n) -> int:
    return load().gs_densify_workspace_size(n)


def gs_densify(params, exp_avg, exp_avg_sq, n, densify_stat, grad_threshold, log_scale_threshold, normals, outs,
               out_stride, workspace, counts, sync=False, stream=None):
    """outs: (params_out, exp_avg_out, exp_avg_sq_out) or None (count only).  Returns the host
    counts (output, clones, splits) when sync=True, else None (they stay in counts)."""
    host = (C.c_int64 * 3)()
    po, mo, vo = outs if outs is not None else (None, None, None)
    _check(load().gs_densify(_ptr(params), _ptr(exp_avg), _ptr(exp_avg_sq), n, _ptr(densify_stat), grad_threshold,
                             log_scale_threshold, _ptr(normals), _ptr(po), _ptr(mo), _ptr(vo), out_stride,
                             _ptr(workspace), workspace.numel() if workspace is not None else 0, _ptr(counts),
                             C.cast(host, C.c_void_p) if sync else None, _stream(stream)), "gs_densify")
    return tuple(host) if sync else None


def gs_probe_ffma(out, blocks, iters, stream=None):
    _check(load().gs_probe_ffma(_ptr(out), blocks, iters, _stream(stream)), "gs_probe_ffma")


def gs_debug_set_wait_limit(iterations: int):
    load().gs_debug_set_wait_limit(iterations)


def gs_debug_drop_publish(mode: int):
    """0 disarms; 1 drops CTA 0's first barrier arrival in the tile sort, 2 in the depth sort."""
    load().gs_debug_drop_publish(int(mode))
