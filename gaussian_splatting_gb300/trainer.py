"""One 3D Gaussian Splatting training step on one GPU, driven through libgs.so.

``Trainer`` owns the device state (parameters, gradients, Adam moments, per-view scratch) as
torch tensors -- torch supplies memory and the stream, every computation is a libgs.so kernel
-- and issues, per batch, the calls of the step in the order of the Grendel-GS training flow
(训练流程): project every view (gs_project_batch), bin/sort them all (gs_bin_sort_batch: the views'
depth sorts share one launch), then for each view composite -> loss -> composite backward (both
compositing calls issue their tiles heaviest first, gs_tile_order); then the visible sets, and
the projection backward of every view with the visible-only Adam update (Odin summary, 研究背景与动机;
Grendel-GS notes §4.2 batch scaling) in one fused pass (gs_project_bwd_adam) whose gradients
never leave the chip. ``step_async(..., adam=False)`` runs the per-view gs_project_bwd instead
and leaves the summed gradients in ``grads``.

The step never synchronises with the host. The tile-instance buffers have a capacity; when a
view overflows it, the update skips itself (it reads the per-view status words), ``step``
notices on its one readback of the loss, grows the buffers and runs the batch again.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

import torch

from . import _native as N

# kernels each entry point launches (memset nodes are not counted)
# (gs_visible_sets given the projection's bitsets: count, scan, offsets, write, intersections,
# Jaccard; the bitset kernel is not launched)
LAUNCHES = {"project": 1, "render_fwd": 1, "loss": 2, "render_bwd": 1, "project_bwd": 1, "visible_sets": 6,
            "sparse_adam": 1, "project_bwd_adam": 1, "tile_order": 1}


MAX_FUSED_BATCH = 16  # views gs_project_bwd_adam takes in one call

# edge of the square blocks of tiles that gs_tile_order ranks together (forward, backward):
# single tiles measured fastest for both (blocks keep more Gaussians shared in L2, but the
# kernels are issue-bound and lose more to the coarser schedule)
ORDER_BLOCK = (1, 1)


def tile_group(views: int, capacity: int) -> int:
    """Views whose tile sorts share one launch in gs_bin_sort_batch: as many as have their own
    capacity-sized ping-pong buffers (16 B per instance) within 1 GiB, 1..8."""
    per_view = 16.0 * max(capacity, 1) + 1024.0 * ((capacity + 3071) // 3072)
    fit = min(8, int(math.floor(float(1 << 30) / per_view)))
    return max(1, min(fit, views, 8))


def bin_sort_launches(views: int, capacity: int) -> int:
    # per group of up to 8 views: zeroing, the depth sorts (keys, the four passes and the
    # tiles-touched scans in one cooperative launch), the tile sorts (both passes of tile_group
    # views per cooperative launch), ranges
    total = 0
    for g0 in range(0, views, 8):
        gv = min(8, views - g0)
        tg = tile_group(views, capacity)
        total += 3 + (gv + tg - 1) // tg
    return total


@dataclasses.dataclass
class StepResult:
    loss: torch.Tensor       # device scalar (float32)
    status: torch.Tensor     # device int64 [B, 2]: instance count and status per view


class Trainer:
    def __init__(self, params: torch.Tensor, width: int, height: int, batch: int, lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-15, w_l1: float = 0.8, w_ssim: float = 0.2,
                 bg=(0.0, 0.0, 0.0), capacity: int = 0, keep_views: bool = False):
        if params.device.type != "cuda" or params.dtype != torch.float32 or params.dim() != 3 or params.shape[0] != 15 \
                or params.shape[2] != 4:
            raise ValueError("params must be a CUDA float32 tensor of shape [15, N, 4]")
        N.load()
        dev = params.device
        self.n = params.shape[1]
        self.width, self.height, self.batch = width, height, batch
        self.lr, self.betas, self.eps = lr, betas, eps
        self.w_l1, self.w_ssim, self.bg = w_l1, w_ssim, tuple(bg)
        self.params = params.contiguous()
        self.grads = torch.zeros_like(self.params)
        self.exp_avg = torch.zeros_like(self.params)
        self.exp_avg_sq = torch.zeros_like(self.params)
        # densification statistic (sum of screen-space mean-gradient lengths, views), gathered by
        # every training step's projection backward and read by densify()
        self.dstat = torch.zeros((self.n, 2), dtype=torch.float32, device=dev)
        self.t = 0
        n, P = self.n, width * height
        tiles = ((width + 15) // 16) * ((height + 15) // 16)
        f32, i32, i64 = torch.float32, torch.int32, torch.int64
        self.proj = torch.zeros((batch, 3, n, 4), dtype=f32, device=dev)
        self.grad2d = torch.zeros((batch, n, 12), dtype=f32, device=dev)  # per view
        self.image = torch.zeros((3, height, width), dtype=f32, device=dev)
        self.T_final = torch.zeros((height, width), dtype=f32, device=dev)
        self.n_contrib = torch.zeros((height, width), dtype=i32, device=dev)
        self.dimg = torch.zeros((3, height, width), dtype=f32, device=dev)
        # keep_views: every view of a step keeps its own image and image gradient (for
        # inspection); otherwise the views share one buffer of each
        self.images = torch.zeros((batch, 3, height, width), dtype=f32, device=dev) if keep_views else None
        self.dimgs = torch.zeros((batch, 3, height, width), dtype=f32, device=dev) if keep_views else None
        self.ranges = torch.zeros((batch, tiles, 2), dtype=i32, device=dev)  # per view
        # launch order of the compositing calls' tiles, heaviest first: [0] for the forward (by
        # list length), [1] for the backward (by the forward's per-tile walk, tile_cost)
        self.tiles_x, self.tiles_y = (width + 15) // 16, (height + 15) // 16
        self.tile_order = torch.zeros((2, tiles), dtype=i32, device=dev)
        self.tile_cost = torch.zeros(tiles, dtype=i32, device=dev)
        self.counts = torch.zeros((batch, 2), dtype=i64, device=dev)
        self.loss = torch.zeros(1, dtype=f32, device=dev)
        self.loss_ws = torch.empty(max(N.gs_loss_workspace_size(width, height), 256), dtype=torch.uint8, device=dev)
        self.vis_ws = torch.empty(max(N.gs_visible_sets_workspace_size(batch, n), 256), dtype=torch.uint8, device=dev)
        # the views' visibility bitsets, written by the batched projection and read by the
        # visible sets and the fused update instead of every view's radius words
        self.bits_stride = max((n + 31) // 32, 1)
        self.vis_bits = torch.zeros((batch, self.bits_stride), dtype=i32, device=dev)
        self.offsets = torch.zeros(batch + 1, dtype=i64, device=dev)
        self.indices = torch.zeros(max(batch * n, 1), dtype=i32, device=dev)
        self.union_idx = torch.zeros(max(n, 1), dtype=i32, device=dev)
        self.n_union = torch.zeros(1, dtype=i64, device=dev)
        self.inter = torch.zeros((batch, batch), dtype=i64, device=dev)
        self.jaccard = torch.zeros((batch, batch), dtype=f32, device=dev)
        self.target_dev = torch.zeros((batch, 3, height, width), dtype=f32, device=dev)
        self.capacity = 0
        self.vals = self.sort_ws = None
        self.copy_stream = None
        self.host_out = None
        self._cam_cache = {}
        self.launches = 0
        self.timer = None  # list of (name, start event, end event) when timing per call
        self.work = None   # list of per-view work counts when measuring (synchronises)
        if capacity:
            self._alloc_sort(capacity)

    # ------------------------------------------------------------------ buffers
    def _alloc_sort(self, capacity: int):
        capacity = int(min(capacity, (1 << 30) - 1))
        dev = self.params.device
        # the sorted keys are not requested: rendering reads the values and the tile ranges
        # (one set per view: the views are sorted together before any is composited)
        self.vals = torch.empty((self.batch, capacity), dtype=torch.int32, device=dev)
        self._ws_cam = None
        self.capacity = capacity
        self.sort_ws = None

    def _camera(self, cam):
        """gs_camera struct of a camera, converted once per distinct camera (keyed by content)."""
        if isinstance(cam, N.Camera):
            return cam
        key = (np.asarray(cam.R, np.float32).tobytes(), np.asarray(cam.t, np.float32).tobytes(), cam.fx, cam.fy,
               cam.cx, cam.cy, cam.znear, cam.width, cam.height)
        hit = self._cam_cache.get(key)
        if hit is None:
            if len(self._cam_cache) > 4096:
                self._cam_cache.clear()
            hit = self._cam_cache[key] = N.camera(cam)
        return hit

    def _sort_ws(self, cam):
        # every view of a trainer has the same image size: the size depends on the capacity only
        # (sized for a full batch, which also covers a single view)
        if self._ws_cam != self.capacity:
            self._ws_need = N.gs_bin_sort_batch_workspace_size(self.batch, self.n, self.capacity, [cam] * self.batch)
            self._ws_cam = self.capacity
        need = self._ws_need
        if self.sort_ws is None or self.sort_ws.numel() < need:
            self.sort_ws = torch.empty(need, dtype=torch.uint8, device=self.params.device)
        return self.sort_ws

    def reserve(self, cams, slack: float = 1.25):
        """Size the instance buffers for these cameras (one synchronising count per view)."""
        best = 0
        for cam in cams:
            N.gs_project(self.params, self.n, cam, self.proj[0])
            if self.capacity == 0:
                self._alloc_sort(1024)
            ws = self._sort_ws(cam)
            try:
                m = N.gs_bin_sort(self.proj[0], self.n, cam, ws, ws.numel(), None, self.vals[0], self.capacity,
                                  self.ranges[0], self.counts[0], sync=True)
            except N.GSError as e:
                if e.status != N.GS_ERR_CAPACITY:
                    raise
                m = int(self.counts[0, 0].item())
            best = max(best, m)
        want = int(best * slack) + 4096
        if want > self.capacity:
            self._alloc_sort(want)
        return best

    def render(self, cam, out: torch.Tensor | None = None, params: torch.Tensor | None = None) -> torch.Tensor:
        """Forward render of one view (project, bin/sort, composite) into ``out`` [3, H, W]."""
        if self.capacity == 0:
            self.reserve([cam])
        params = self.params if params is None else params
        if out is None:
            out = torch.empty((3, self.height, self.width), dtype=torch.float32, device=self.params.device)
        proj = self.proj[0]
        N.gs_project(params, self.n, cam, proj)
        ws = self._sort_ws(cam)
        N.gs_bin_sort(proj, self.n, cam, ws, ws.numel(), None, self.vals[0], self.capacity, self.ranges[0],
                      self.counts[0])
        N.gs_tile_order(self.ranges[0], None, self.tiles_x, self.tiles_y, self.tile_order[0], block=ORDER_BLOCK[0])
        N.gs_render_fwd(proj, self.n, self.vals[0], self.ranges[0], cam, self.bg, out, self.T_final, self.n_contrib,
                        tile_order=self.tile_order[0])
        return out

    def prune(self, min_opacity: float) -> int:
        """Drop the Gaussians whose opacity is below ``min_opacity`` (the pruning half of
        densification): parameters and Adam moments are compacted in index order by gs_prune,
        the per-Gaussian scratch is resized, the gradients start from zero.  Synchronises;
        returns the new count."""
        if min_opacity <= 0.0:
            logit = -math.inf
        elif min_opacity >= 1.0:
            logit = math.inf
        else:
            logit = math.log(min_opacity / (1.0 - min_opacity))
        dev, n = self.params.device, self.n
        ws = torch.empty(max(N.gs_prune_workspace_size(n), 256), dtype=torch.uint8, device=dev)
        nk = torch.zeros(1, dtype=torch.int64, device=dev)
        sets = [self.params, self.exp_avg, self.exp_avg_sq]
        k = N.gs_prune(sets, n, logit, None, 0, ws, nk, sync=True)  # the count
        outs = [torch.empty((15, k, 4), dtype=torch.float32, device=dev) for _ in sets]
        if k > 0:
            N.gs_prune(sets, n, logit, outs, k, ws, nk, sync=True)
        self.params, self.exp_avg, self.exp_avg_sq = outs
        self._alloc_gaussians(k)
        return k

    def densify(self, grad_threshold: float, scale_threshold: float, seed: int = 0):
        """Clone / split (the growing half of densification) by gs_densify: the Gaussians whose
        mean screen-space mean-gradient length over the views that saw them since the last
        densify() reaches grad_threshold are cloned, or split in two if their largest scale
        exceeds scale_threshold (world units); the children's offsets use standard normals
        drawn from `seed`.  New Gaussians start with zero moments, the statistic and the
        gradients restart from zero.  Synchronises; returns (count, clones, splits)."""
        dev, n = self.params.device, self.n
        gen = torch.Generator(device=dev)
        gen.manual_seed(int(seed))
        normals = torch.randn((max(n, 1), 6), generator=gen, device=dev, dtype=torch.float32)
        ws = torch.empty(max(N.gs_densify_workspace_size(n), 256), dtype=torch.uint8, device=dev)
        counts = torch.zeros(3, dtype=torch.int64, device=dev)
        lthr = math.log(scale_threshold) if scale_threshold > 0 else -math.inf
        total, clones, splits = N.gs_densify(self.params, self.exp_avg, self.exp_avg_sq, n, self.dstat,
                                             grad_threshold, lthr, normals, None, 0, ws, counts, sync=True)
        outs = [torch.empty((15, max(total, 1), 4), dtype=torch.float32, device=dev) for _ in range(3)]
        if total > 0:
            N.gs_densify(self.params, self.exp_avg, self.exp_avg_sq, n, self.dstat, grad_threshold, lthr, normals,
                         outs, total, ws, counts, sync=True)
        self.params, self.exp_avg, self.exp_avg_sq = (o[:, :total] if total else o[:, :0] for o in outs)
        self.params = self.params.contiguous()
        self.exp_avg = self.exp_avg.contiguous()
        self.exp_avg_sq = self.exp_avg_sq.contiguous()
        self._alloc_gaussians(total)
        return total, clones, splits

    def _alloc_gaussians(self, n: int):
        """(Re)allocate the per-Gaussian scratch for n Gaussians."""
        dev, batch = self.params.device, self.batch
        f32, i32 = torch.float32, torch.int32
        self.n = n
        self.grads = torch.zeros_like(self.params)
        self.dstat = torch.zeros((n, 2), dtype=f32, device=dev)
        self.proj = torch.zeros((batch, 3, n, 4), dtype=f32, device=dev)
        self.grad2d = torch.zeros((batch, n, 12), dtype=f32, device=dev)
        self.vis_ws = torch.empty(max(N.gs_visible_sets_workspace_size(batch, n), 256), dtype=torch.uint8, device=dev)
        self.bits_stride = max((n + 31) // 32, 1)
        self.vis_bits = torch.zeros((batch, self.bits_stride), dtype=i32, device=dev)
        self.indices = torch.zeros(max(batch * n, 1), dtype=i32, device=dev)
        self.union_idx = torch.zeros(max(n, 1), dtype=i32, device=dev)
        self.sort_ws = None
        self._ws_cam = None

    # ------------------------------------------------------------------ the step
    def _timed(self, name, fn, *args, **kw):
        if self.timer is None:
            return fn(*args, **kw)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        fn(*args, **kw)
        e.record()
        self.timer.append((name, s, e))

    def _enqueue(self, cams, targets: torch.Tensor, adam: bool = True, ready=None, host_targets=None):
        B = len(cams)
        n, W, H = self.n, self.width, self.height
        inv_b = 1.0 / B
        launches = 0
        T = self._timed
        fused = adam and B <= MAX_FUSED_BATCH
        # marshal once per step: the cameras as gs_camera structs, the stream as a handle
        ccams = [self._camera(c) for c in cams]
        st = torch.cuda.current_stream().cuda_stream
        step_start = None
        if host_targets is not None:  # marks the point the target uploads may start from
            step_start = torch.cuda.Event()
            step_start.record()
        T("project", N.gs_project_batch, self.params, n, ccams, [self.proj[b] for b in range(B)], stream=st,
          visible_bits=self.vis_bits, bits_stride=self.bits_stride)
        ws = self._sort_ws(ccams[0])
        T("bin_sort", N.gs_bin_sort_batch, [self.proj[b] for b in range(B)], n, ccams, ws, ws.numel(), None,
          [self.vals[b] for b in range(B)], self.capacity, [self.ranges[b] for b in range(B)], self.counts,
          stream=st)
        launches += (B + 15) // 16 * LAUNCHES["project"] + bin_sort_launches(B, self.capacity)
        for b, cam in enumerate(ccams):
            proj, vals, ranges = self.proj[b], self.vals[b], self.ranges[b]
            image = self.image if self.images is None else self.images[b]
            dimg = self.dimg if self.dimgs is None else self.dimgs[b]
            work_buf = None
            if self.work is not None:
                work_buf = torch.zeros((3, H, W), dtype=torch.int32, device=self.params.device)
            T("tile_order", N.gs_tile_order, ranges, None, self.tiles_x, self.tiles_y, self.tile_order[0],
              block=ORDER_BLOCK[0], stream=st)
            T("render_fwd", N.gs_render_fwd, proj, n, vals, ranges, cam, self.bg, image, self.T_final,
              self.n_contrib, work_buf, stream=st, tile_order=self.tile_order[0], tile_cost=self.tile_cost)
            if host_targets is not None and ready is None:  # after the first view's compositing
                ready = self._upload(host_targets, B, step_start)
            if ready is not None:
                torch.cuda.current_stream().wait_event(ready[b])
            T("loss", N.gs_loss, image, targets[b], W, H, self.w_l1, self.w_ssim, inv_b, self.loss, b > 0,
              dimg, self.loss_ws, self.loss_ws.numel(), stream=st)
            T("tile_order", N.gs_tile_order, None, self.tile_cost, self.tiles_x, self.tiles_y, self.tile_order[1],
              block=ORDER_BLOCK[1], stream=st)
            T("render_bwd", N.gs_render_bwd, proj, n, vals, ranges, cam, self.bg, self.T_final,
              self.n_contrib, dimg, self.grad2d[b], stream=st, tile_order=self.tile_order[1])
            if not fused:
                T("project_bwd", N.gs_project_bwd, self.params, n, cam, proj, self.grad2d[b], self.grads,
                  self.dstat if adam else None, stream=st)
                launches += LAUNCHES["project_bwd"]
            if self.work is not None:
                # (entries evaluated in the forward, entries accumulated, entries walked by the backward,
                #  pairs the forward's warps evaluated)
                self.work.append((int(work_buf[0].sum()), int(work_buf[1].sum()), int(self.n_contrib.sum()),
                                  int(work_buf[2].sum())))
            launches += sum(LAUNCHES[k] for k in ("render_fwd", "loss", "render_bwd")) + 2 * LAUNCHES["tile_order"]
        T("visible_sets", N.gs_visible_sets, [self.proj[b] for b in range(B)], B, n, self.vis_ws, self.vis_ws.numel(),
          self.offsets, self.indices, self.union_idx, self.n_union, self.inter, self.jaccard, stream=st,
          visible_bits=self.vis_bits, bits_stride=self.bits_stride)
        launches += LAUNCHES["visible_sets"]
        if fused:
            T("project_bwd_adam", N.gs_project_bwd_adam, self.params, n, ccams, [self.proj[b] for b in range(B)],
              [self.grad2d[b] for b in range(B)], self.exp_avg, self.exp_avg_sq, self.lr, self.betas[0],
              self.betas[1], self.eps, self.t + 1, self.counts, B, self.dstat, stream=st,
              visible_bits=self.vis_bits, bits_stride=self.bits_stride)  # the projection's bitsets
            launches += LAUNCHES["project_bwd_adam"]
        elif adam:
            T("sparse_adam", N.gs_sparse_adam, self.params, self.grads, self.exp_avg, self.exp_avg_sq, n,
              self.union_idx, self.n_union, n, self.lr, self.betas[0], self.betas[1], self.eps, B, self.t + 1,
              self.counts, B, stream=st)
            launches += LAUNCHES["sparse_adam"]
        self.launches = launches

    def step_async(self, cams, targets: torch.Tensor, adam: bool = True) -> StepResult:
        """Enqueue one step on the current stream without any host synchronisation.

        ``targets`` is a device tensor [B, 3, H, W].  The caller must check ``status``
        (all [:, 1] zero) before trusting the update; ``step`` does that for you.
        """
        return self._step_async(cams, targets, adam, None)

    def _step_async(self, cams, targets, adam, ready, host_targets=None):
        if self.capacity == 0:
            self.reserve(cams)
        self._enqueue(cams, targets, adam, ready, host_targets)
        if adam:
            self.t += 1
        return StepResult(self.loss, self.counts)

    def _upload(self, targets: torch.Tensor, B: int, after: torch.cuda.Event):
        """Copy host targets into target_dev on the side stream once `after` (recorded before the
        step's first kernel) has passed; returns one event per view."""
        if self.copy_stream is None:
            self.copy_stream = torch.cuda.Stream(device=self.params.device)
        cs = self.copy_stream
        cs.wait_event(after)  # target_dev no longer read by earlier steps
        events = []
        with torch.cuda.stream(cs):
            for b in range(B):
                self.target_dev[b].copy_(targets[b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                events.append(ev)
        return events

    def step(self, cams, targets: torch.Tensor, adam: bool = True) -> float:
        """One training step over the views ``cams``; returns the batch loss (host float).

        ``targets`` may be a device tensor or a (pinned) host tensor [B, 3, H, W].  Host
        targets are copied in view by view on a side stream, enqueued once the first view's
        projection, binning and compositing are; view b's loss waits only for its own copy.
        The status words and the loss come back in one synchronisation.
        """
        host = targets if targets.device.type != "cuda" else None
        if host is not None:
            targets = self.target_dev
        if self.host_out is None:
            self.host_out = (torch.empty((self.batch, 2), dtype=torch.int64).pin_memory(),
                             torch.empty(1, dtype=torch.float32).pin_memory())
        # the unfused path (more than 16 views) adds to the statistic before the overflow check
        # can skip anything: keep a copy to restore if the batch has to run again
        dstat0 = self.dstat.clone() if adam and len(cams) > MAX_FUSED_BATCH else None
        while True:
            res = self._step_async(cams, targets, adam, None, host)
            host = None  # a re-run reuses the uploaded targets
            hc, hl = self.host_out
            hc.copy_(res.status, non_blocking=True)
            hl.copy_(res.loss, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            counts = hc
            if int(counts[: len(cams), 1].abs().sum()) == 0:
                return float(hl[0])
            if adam:
                self.t -= 1
            if int(counts[:, 1].bitwise_and(2).sum()) != 0:
                raise RuntimeError("gs_bin_sort: a device-side wait gave up")
            # overflow: the update was skipped; clear the partial gradients and grow
            self.grads.zero_()
            if dstat0 is not None:
                self.dstat.copy_(dstat0)
            self._alloc_sort(int(int(counts[:, 0].max()) * 1.25) + 4096)
