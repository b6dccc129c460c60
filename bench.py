"""Benchmark: train views/s of the 3D Gaussian Splatting training step (fwd + bwd + Adam).

Workload (default, ``--config 4``): the largest single-GPU scene, 40M Gaussians in a city
layout of 1024 box clusters, 3840x2160 views, batch 16, 64 views on an orbit, all fp32,
seeded synthetic data (scene generator in scenes/).  ``--config 1`` is the 300K-Gaussian
object scene at 1236x820, batch 4.  One step = one batch of views: projection, binning +
radix sort of every view, then per view compositing, L1 + D-SSIM loss and compositing
backward; then the visible sets and the projection backward with the visible-only Adam
update.  throughput = steps * batch / time.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
Targets are rendered (untimed) by the CUDA path from means jittered by N(0, 0.02).
Between timed steps L2 is flushed by writing a 512 MB buffer (outside the timed events).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import scenes  # noqa: E402

METRIC = "train views/s (fwd+bwd+Adam) at N Gaussians x res; % of HBM/FP32 roofline"
UNIT = "views/s"

# Algorithmic flops per unit of work (FMA = 2): per pixel-Gaussian pair that the pixel itself
# evaluates through its termination point, 15 for the forward compositing and 40 for the
# backward (plus one ex2 each, not counted); about 1.3 kflop per pixel for the loss
# (5 statistics x 2 passes x 11 taps x 2 flops x 3 channels forward, as much again backward).
FWD_FLOPS_PER_PAIR = 15
BWD_FLOPS_PER_PAIR = 40
LOSS_FLOPS_PER_PIXEL = 1320
# FP32 lanes per SM of this architecture (4 sub-partitions x 32); the peak is derived from the
# device's SM count and its maximum SM clock (FMA = 2 flops)
FP32_LANES_PER_SM = 128
HBM_FALLBACK_GBS = 6800.0

# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one ncu capture,
# keyed by entry point and workload, valid only for the kernel source it was measured on: when
# the source file's hash differs the figure is reported as null.  (The render_bwd figures were
# taken on this backward kernel; since then the tile-order kernel left the file and the
# forward kernel's transmittance update and finished-pixel parking changed.)
NCU_TRAFFIC = {
    # one launch on the 300K-Gaussian 1236x820 view (tiles issued heaviest first): 38.226 MB
    # read + 0.077 MB written
    ("render_bwd", "object-300k-1236x820"): {"source": "gaussian_splatting_gb300/csrc/render.cu",
                                             "sha256": "32cf7c6a3f1dcace3465f1b26b0f0de88dece516b54b1115aa70d1feabfd7b7c",
                                             "bytes": 38302976},
    # one launch on a 10M-Gaussian 3840x2160 view of the city layout (55.2M instances, tiles
    # issued heaviest first): 5.055 GB read + 0.392 GB written, scaled by the instances to the
    # 40M view's 216.2M (x 3.914)
    ("render_bwd", "city-40m-3840x2160"): {"source": "gaussian_splatting_gb300/csrc/render.cu",
                                           "sha256": "32cf7c6a3f1dcace3465f1b26b0f0de88dece516b54b1115aa70d1feabfd7b7c",
                                           "bytes": 21320000000, "scaled_from": "10M-Gaussian capture, by instances"},
}


def fp32_peak_tflops(sm_count: int, sm_max_mhz: float) -> float:
    return sm_count * FP32_LANES_PER_SM * 2 * sm_max_mhz * 1e6 / 1e12


def max_sm_mhz(gpu_index: int) -> float:
    """Maximum SM clock reported by nvidia-smi (2070 MHz on GB300 if it cannot be read)."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=clocks.max.sm",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20).stdout
        return float(out.strip().splitlines()[0])
    except Exception:
        return 2070.0


def measured_traffic(name, workload):
    import hashlib
    rec = NCU_TRAFFIC.get((name, workload))
    if not rec or not rec["sha256"] or rec["bytes"] is None:
        return None
    path = os.path.join(ROOT, rec["source"])
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return rec["bytes"] if digest == rec["sha256"] else None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as fh:
                return json.load(fh), "measured"
        except Exception:
            pass
    return {}, "fallback"


def hbm_peak():
    d, src = measured_peaks()
    for k in ("hbm_gbs", "hbm_GBs", "hbm"):
        if k in d and isinstance(d[k], (int, float)):
            return float(d[k]), src
    return HBM_FALLBACK_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------- oracle timing
def _reach(P, cam):
    """Screen position and a bound on the reach of every Gaussian's tile rectangle in a view:
    r = ceil(3 sqrt(lambda_max)) <= 3 sqrt((f/z)^2 (2 + xr^2 + yr^2) s_max^2 + 0.3) + 1, and the
    rectangle's tile rounding adds at most 17 pixels.  Returns (u, v, reach, in front)."""
    R = np.asarray(cam.R, np.float64)
    t = np.asarray(cam.t, np.float64)
    limx = 1.3 * (cam.width / 2.0) / cam.fx
    limy = 1.3 * (cam.height / 2.0) / cam.fy
    out = []
    for a in range(0, P.shape[1], 4_000_000):  # chunks bound the float64 temporaries
        pc = P[0, a:a + 4_000_000, :3].astype(np.float64) @ R.T + t
        z = pc[:, 2]
        front = z > 0.99 * cam.znear
        zs = np.where(front, z, 1.0)
        xr = np.clip(pc[:, 0] / zs, -limx, limx)
        yr = np.clip(pc[:, 1] / zs, -limy, limy)
        smax = np.exp(P[1, a:a + 4_000_000, :3].astype(np.float64).max(axis=1))
        lam = (max(cam.fx, cam.fy) / zs) ** 2 * (2.0 + xr * xr + yr * yr) * smax * smax + 0.3
        r = 3.0 * np.sqrt(lam) + 18.0
        u = cam.fx * pc[:, 0] / zs + cam.cx
        v = cam.fy * pc[:, 1] / zs + cam.cy
        out.append((u.astype(np.float32), v.astype(np.float32), r.astype(np.float32), front))
    return tuple(np.concatenate([o[k] for o in out]) for k in range(4))


def _band_reach(info, width, r0, rows):
    """Indices of every Gaussian whose tile rectangle can meet rows [r0, r0 + rows) (a
    superset), so that the band's camera renders the same image from them alone as from the
    whole scene.  (The band's camera is the view's with the principal point moved up by r0 and
    an image `rows` high: its field of view, and with it the 1.3 tan(fov/2) clamp of the
    projection's Jacobian in y, is the band's, so its image is close to, not equal to, those
    rows of the whole view: a sample of the view's work, not of its pixels.)"""
    u, v, r, front = info
    hit = front & (u + r >= 0) & (u - r <= width) & (v + r >= r0) & (v - r <= r0 + rows)
    return np.nonzero(hit)[0]


def _oracle_worker(conn, P, jit, cam, lr, eps):
    """One host core's share of the CPU baseline: the oracle's whole step (project, bin,
    composite, loss, backward, Adam) on its band, once per request.  The band's target is
    the oracle's render of the jittered scene (untimed)."""
    import oracle

    tgt = oracle.render_view(jit, cam)[None]
    zeros = np.zeros_like(P)
    conn.send("ready")
    while conn.recv() == "go":
        t0 = time.perf_counter()
        oracle.step(P, zeros, zeros, [cam], tgt, lr=lr, eps=eps)
        conn.send(time.perf_counter() - t0)
    conn.close()


def available_host_bytes() -> int:
    """MemAvailable of /proc/meminfo (64 GB if it cannot be read)."""
    try:
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 64 << 30


class OracleSampler:
    """Times the CPU oracle, as it stands, on the host cores: one spawned process per core (as
    many as the host memory holds), each running the oracle's whole step (batch 1) on its own
    band of `rows` image rows at full width (one band in the middle of each equal share of view
    0's rows, then of the next views), on the Gaussians that can reach the band.  One round =
    every process takes one step; throughput = (bands x rows / height) views / wall time of the
    round."""

    # host memory the oracle's step holds per Gaussian it is given (double-precision parameters,
    # moments and gradients, and its per-Gaussian records): a worker's peak resident set on a
    # 16-row band of the 4K view is 4.8 KB per Gaussian; with slack
    BYTES_PER_GAUSSIAN = 5500
    MAX_BAND_GAUSSIANS = 1_500_000

    def __init__(self, cfg_idx: int, P=None, cams=None, jit=None, workers: int | None = None):
        self.cfg = scenes.CONFIGS[cfg_idx]
        self.P = scenes.make_params(cfg_idx) if P is None else P
        self.cams = scenes.make_cameras(cfg_idx) if cams is None else cams
        self.jit = scenes.jitter_means(self.P, self.cfg.jitter, 2000 + cfg_idx) if jit is None else jit
        self.workers = workers or max(1, len(os.sched_getaffinity(0)))
        self.rows = None
        self.procs = []
        self._info = {}

    def _band_idx(self, k):
        """Band k: its camera, its height and the indices of the Gaussians that can reach it."""
        H = self.cfg.height
        # the processes' bands spread evenly over the image height, each in the middle of its
        # equal share of the rows (the content of a view is not uniform: the top rows of a city
        # view see little, so a band at the top of each share would favour the empty sky), then
        # over the next views
        per_view = max(1, min(H // self.rows, self.workers))
        view = (k // per_view) % len(self.cams)
        mid = (2 * (k % per_view) + 1) * H // (2 * per_view)
        r0 = min(max(0, mid - self.rows // 2) // 16 * 16, max(0, H - self.rows) // 16 * 16)
        rows = min(self.rows, H - r0)
        c = self.cams[view]
        cam = scenes.Camera(c.R, c.t, c.fx, c.fy, c.cx, c.cy - r0, c.znear, c.width, rows)
        if view not in self._info:
            self._info[view] = _reach(self.P, c)
        return cam, rows, _band_reach(self._info[view], c.width, r0, rows)

    def _band(self, k):
        cam, rows, idx = self._band_idx(k)
        return self.P[:, idx], self.jit[:, idx], cam, rows

    def calibrate(self, budget_s: float):
        """Band height (a multiple of 16) whose step takes about budget_s on one core, and at
        most as tall as keeps a band's Gaussians within MAX_BAND_GAUSSIANS."""
        import oracle

        self.rows = 16
        P, jit, cam, rows = self._band(self.workers // 2)  # a band in the middle of the view
        tgt = oracle.render_view(jit, cam)[None]
        t0 = time.perf_counter()
        oracle.step(P, np.zeros_like(P), np.zeros_like(P), [cam], tgt, lr=self.cfg.lr, eps=self.cfg.eps)
        t16 = max(time.perf_counter() - t0, 1e-3)
        del P, jit, tgt
        self.rows = int(max(16, min(self.cfg.height, 16 * math.floor(budget_s / t16))))
        self.rows = max(16, self.rows // 16 * 16)
        while self.rows > 16 and self._largest_band() > self.MAX_BAND_GAUSSIANS:
            self.rows = max(16, (self.rows // 2) // 16 * 16)
        return self.rows

    def _largest_band(self):
        return max(len(self._band_idx(k)[2]) for k in range(self.workers))

    def start(self):
        import multiprocessing as mp

        # as many processes as host cores, and as the available memory holds (a band is made,
        # handed to its process and dropped before the next one)
        need = self._largest_band() * self.BYTES_PER_GAUSSIAN
        fit = max(1, int(0.5 * available_host_bytes() // max(need, 1)))
        self.workers = min(self.workers, fit)
        ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
        for k in range(self.workers):
            P, jit, cam, rows = self._band(k)
            a, b = ctx.Pipe()
            pr = ctx.Process(target=_oracle_worker, args=(b, P, jit, cam, self.cfg.lr, self.cfg.eps), daemon=True)
            pr.start()
            self.procs.append((pr, a, rows))
            del P, jit
        for _, a, _ in self.procs:
            assert a.recv() == "ready"

    def round(self):
        """One timed round: (views/s, wall seconds, views)."""
        t0 = time.perf_counter()
        for _, a, _ in self.procs:
            a.send("go")
        for _, a, _ in self.procs:
            a.recv()
        wall = time.perf_counter() - t0
        views = sum(rows for _, _, rows in self.procs) / self.cfg.height
        return views / wall, wall, views

    def stop(self):
        for pr, a, _ in self.procs:
            try:
                a.send("stop")
            except Exception:
                pass
            pr.join(timeout=30)
        self.procs = []

    def describe(self, wall):
        return (f"{self.workers} processes (one per host core, as many as half the free host memory holds), "
                f"each the oracle's whole step (project, bin, composite, loss, backward, Adam; batch 1, double "
                f"precision) on its own band of {self.rows} rows at full width (one band in the middle of each "
                f"equal share of view 0's height, then of the next views) with the Gaussians that can reach it; "
                f"{wall:.1f} s per round")


# ---------------------------------------------------------------------- main
def rank_views(step: int, rank: int, world: int, batch: int, n_views: int) -> list[int]:
    """The views rank `rank` trains in step `step`: consecutive batches dealt round-robin over
    the ranks (replicas: every rank its own views, no exchange)."""
    return [((step * world + rank) * batch + b) % n_views for b in range(batch)]


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over the ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


_T0 = time.perf_counter()


def log(msg: str):
    """Progress on stderr (the JSON line alone goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def kernels_mode(args):
    """One view of the workload's first camera (project, bin and sort, composite, loss,
    composite backward), every call timed on its own with CUDA events (best of --steps after
    --warmup).  The scene can be drawn smaller (--gaussians) and the calls limited (--calls) so
    that a profiler capture holds a few GB on the device.  Prints one JSON line of per-call
    milliseconds."""
    import torch
    from gaussian_splatting_gb300 import _native as N
    from gaussian_splatting_gb300.trainer import ORDER_BLOCK

    cfg = scenes.CONFIGS[args.config]
    n = args.gaussians or cfg.n
    P = scenes.make_params(args.config, n=n)
    cam = scenes.make_cameras(args.config)[0]
    W, H = cam.width, cam.height
    Pd = torch.from_numpy(P).cuda()
    proj = torch.zeros((3, n, 4), dtype=torch.float32, device="cuda")
    N.gs_project(Pd, n, cam, proj)
    torch.cuda.synchronize()
    M = int(proj[2, :, 3].contiguous().view(torch.int32).long().sum())
    cap = M + 4096
    vals = torch.empty(cap, dtype=torch.int32, device="cuda")
    ranges = torch.zeros((cam.tiles_x * cam.tiles_y, 2), dtype=torch.int32, device="cuda")
    counts = torch.zeros((1, 2), dtype=torch.int64, device="cuda")
    wsb = N.gs_bin_sort_batch_workspace_size(1, n, cap, [cam])
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    img = torch.empty((3, H, W), device="cuda")
    Tf = torch.empty((H, W), device="cuda")
    nc = torch.empty((H, W), dtype=torch.int32, device="cuda")
    gen = torch.Generator(device="cuda")
    gen.manual_seed(3000 + args.config)
    tgt = torch.rand((3, H, W), device="cuda", generator=gen)
    dimg = torch.empty((3, H, W), device="cuda")
    lws = torch.empty(N.gs_loss_workspace_size(W, H), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(1, device="cuda")
    g2d = torch.zeros((n, 12), device="cuda")
    T = cam.tiles_x * cam.tiles_y
    order = torch.zeros((2, T), dtype=torch.int32, device="cuda")
    tcost = torch.zeros(T, dtype=torch.int32, device="cuda")
    per_view = {
        "project": lambda: N.gs_project(Pd, n, cam, proj),
        "bin_sort": lambda: N.gs_bin_sort_batch([proj], n, [cam], ws, wsb, None, [vals], cap, [ranges], counts),
        "tile_order_fwd": lambda: N.gs_tile_order(ranges, None, cam.tiles_x, cam.tiles_y, order[0],
                                                  block=ORDER_BLOCK[0]),
        "render_fwd": lambda: N.gs_render_fwd(proj, n, vals, ranges, cam, None, img, Tf, nc, tile_order=order[0],
                                              tile_cost=tcost),
        "loss": lambda: N.gs_loss(img, tgt, W, H, 0.8, 0.2, 1.0, loss, False, dimg, lws, lws.numel()),
        "tile_order_bwd": lambda: N.gs_tile_order(None, tcost, cam.tiles_x, cam.tiles_y, order[1],
                                                  block=ORDER_BLOCK[1]),
        "render_bwd": lambda: N.gs_render_bwd(proj, n, vals, ranges, cam, None, Tf, nc, dimg, g2d,
                                              tile_order=order[1]),
    }
    # one untimed pass of the view's calls prepares every call's inputs; --calls keeps only the
    # named ones (and the buffers they need: a profiler capture then holds less)
    for f in per_view.values():
        f()
    want = set(args.calls.split(",")) if args.calls else None
    calls = {k: f for k, f in per_view.items() if want is None or k in want}
    if want is None or "project_bwd_adam" in want:
        # the batch's fused projection backward + Adam, every view with its own projection and
        # a copy of view 0's screen-space gradients
        B = min(cfg.batch, 16)
        bcams = scenes.make_cameras(args.config)[:B]
        bprojs = [torch.zeros((3, n, 4), dtype=torch.float32, device="cuda") for _ in range(B)]
        N.gs_project_batch(Pd, n, bcams, bprojs)
        g2ds = [g2d.clone() for _ in range(B)]
        m_, v_ = torch.zeros_like(Pd), torch.zeros_like(Pd)
        Pu = Pd.clone()
        stat = torch.zeros((n, 2), dtype=torch.float32, device="cuda")
        # the views' visibility bitsets, as the trainer hands them over from gs_visible_sets
        vws = torch.empty(N.gs_visible_sets_workspace_size(B, n), dtype=torch.uint8, device="cuda")
        i64 = dict(dtype=torch.int64, device="cuda")
        N.gs_visible_sets(bprojs, B, n, vws, vws.numel(), torch.zeros(B + 1, **i64),
                          torch.zeros(B * n, dtype=torch.int32, device="cuda"),
                          torch.zeros(n, dtype=torch.int32, device="cuda"), torch.zeros(1, **i64),
                          torch.zeros((B, B), **i64), torch.zeros((B, B), dtype=torch.float32, device="cuda"))
        calls["project_bwd_adam"] = lambda: N.gs_project_bwd_adam(Pu, n, bcams, bprojs, g2ds, m_, v_, 1e-3, 0.9,
                                                                  0.999, 1e-15, 1, densify_stat=stat,
                                                                  visible_bits=vws, bits_stride=(n + 31) // 32)
    for _ in range(max(1, args.warmup)):
        for f in calls.values():
            f()
    torch.cuda.synchronize()
    res = {"workload": cfg.name, "gaussians": n, "instances": M, "status": counts.cpu().tolist()}
    for name, f in calls.items():
        best = None
        for _ in range(max(1, args.steps)):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            f()
            b.record()
            torch.cuda.synchronize()
            best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
        res[name + "_ms"] = round(best, 4)
    print(json.dumps(res), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gs", choices=["gs", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--kernels", action="store_true",
                    help="time the stage calls of one view of the workload (for profiler captures)")
    ap.add_argument("--gaussians", type=int, default=0, help="with --kernels: draw this many Gaussians instead")
    ap.add_argument("--calls", default="", help="with --kernels: comma-separated calls to time (default: all)")
    args = ap.parse_args()
    if args.kernels:
        return kernels_mode(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = scenes.CONFIGS[args.config]
    workload = {"workload": cfg.name, "gaussians": cfg.n, "width": cfg.width, "height": cfg.height,
                "batch": cfg.batch, "views": cfg.n_views, "focal": cfg.focal}

    if args.impl == "reference":
        if rank != 0:
            return 0
        # each step is one round of the oracle on every host core (a bounded sample of the
        # workload: one band of rows per core); the rounds are sized so that the whole run
        # takes about two minutes
        smp = OracleSampler(args.config)
        smp.calibrate(max(1.0, 120.0 / max(1, args.steps + args.warmup)))
        smp.start()
        per_step, walls, views = [], [], 0.0
        for i in range(args.warmup + args.steps):
            v, wall, views = smp.round()
            if i >= args.warmup:
                per_step.append(v)
                walls.append(wall)
        smp.stop()
        value = views * len(walls) / sum(walls)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1000.0 * sum(walls) / len(walls), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {**workload, "l2": "n/a (CPU)"}, "impl": "reference",
                "sample_views_per_step": views,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.workers, "kind": "oracle",
                                 "sample": "each step: " + smp.describe(statistics.median(walls))},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    import torch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from gaussian_splatting_gb300 import Trainer
    from gaussian_splatting_gb300 import _native as N

    log(f"workload {cfg.name}: drawing the scene")
    P = scenes.make_params(args.config)
    cams = scenes.make_cameras(args.config)
    jit = scenes.jitter_means(P, cfg.jitter, 2000 + args.config)
    log("scene drawn; rendering the targets")
    params = torch.from_numpy(P).cuda()
    tr = Trainer(params.clone(), cfg.width, cfg.height, cfg.batch, lr=cfg.lr, betas=(cfg.beta1, cfg.beta2),
                 eps=cfg.eps, w_l1=cfg.w_l1, w_ssim=cfg.w_ssim)
    tr.reserve(cams)
    # targets: render of the jittered scene for every view (untimed setup)
    jit_dev = torch.from_numpy(jit).cuda()
    targets = torch.empty((cfg.n_views, 3, cfg.height, cfg.width), dtype=torch.float32, device="cuda")
    for v, cam in enumerate(cams):
        tr.render(cam, targets[v], params=jit_dev)
    torch.cuda.synchronize()
    del jit_dev
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def batch_of(step):
        ids = rank_views(step, rank, world, cfg.batch, cfg.n_views)
        return ids, [cams[i] for i in ids]

    def run_step(step):
        ids, bc = batch_of(step)
        tgt = targets[ids[0]:ids[0] + cfg.batch] if ids == list(range(ids[0], ids[0] + cfg.batch)) \
            else targets[torch.tensor(ids, device="cuda")]
        tr.step_async(bc, tgt)

    log("targets rendered; warm-up")
    for s in range(args.warmup):
        run_step(s)
    torch.cuda.synchronize()
    st = tr.counts.cpu()
    if int(st[:, 1].abs().sum()) != 0:
        raise SystemExit(f"binning overflow during warm-up: {st.tolist()}")

    # ---------------- measured FP32 throughput (FFMA probe), best of three launches
    fp32_meas = None
    try:
        probe_blocks = torch.cuda.get_device_properties(0).multi_processor_count * 8
        probe_out = torch.empty(probe_blocks * 256, dtype=torch.float32, device="cuda")
        best = None
        for _ in range(4):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            N.gs_probe_ffma(probe_out, probe_blocks, 4096)
            b.record()
            torch.cuda.synchronize()
            best = min(best or 1e9, a.elapsed_time(b))
        fp32_meas = probe_blocks * 256 * 4096 * 16 / (best / 1e3) / 1e12
        del probe_out
    except Exception:
        fp32_meas = None

    log("timed steps")
    # ---------------- timed region (device time, CUDA events per step)
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    tr.timer = []
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        torch.cuda.nvtx.range_push("timed")  # profilers select the timed steps by this range
        for s in range(args.steps):
            flush.zero_()
            starts[s].record(stream)
            run_step(args.warmup + s)
            ends[s].record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
    if dist:
        dist.barrier()
    st = tr.counts.cpu()
    if int(st[:, 1].abs().sum()) != 0:
        raise SystemExit(f"binning overflow in the timed region: {st.tolist()}")
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    per_call = {}
    for name, a, b in tr.timer:
        per_call.setdefault(name, []).append(a.elapsed_time(b))
    tr.timer = None
    launches = tr.launches * args.steps
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    views = args.steps * cfg.batch * world
    value = views / (total_ms / 1000.0)

    # ---------------- work counts over exactly one orbit (every view once, the batches the timed
    # steps cycle through), untimed, gradients only: the parameters do not move and the
    # gradients are cleared.  The timed steps weight the views (almost) evenly too.
    tr.work = []
    orbit = (cfg.n_views + cfg.batch * world - 1) // (cfg.batch * world)
    for s in range(orbit):
        ids, bc = batch_of(s)
        tr.step_async(bc, targets[torch.tensor(ids, device="cuda")], adam=False)
        tr.grads.zero_()
    work = tr.work
    tr.work = None
    n_views = max(1, len(work))
    ev = sum(w[0] for w in work) / n_views
    used = sum(w[1] for w in work) / n_views
    walked = sum(w[2] for w in work) / n_views
    warp_pairs = sum(w[3] for w in work) / n_views
    # ---------------- the scheduling helpers on this workload (untimed by the step): Grendel's
    # balanced tile split of one view's per-pixel cost (the entries each pixel's warp walked),
    # and the Odin view order on the batch's Jaccard weights
    schedule = None
    try:
        ids, bc = batch_of(args.warmup + args.steps - 1)
        H, W, B = cfg.height, cfg.width, cfg.batch
        wk = torch.zeros((3, H, W), dtype=torch.int32, device="cuda")
        img = torch.empty((3, H, W), dtype=torch.float32, device="cuda")
        Tf = torch.empty((H, W), dtype=torch.float32, device="cuda")
        nc = torch.empty((H, W), dtype=torch.int32, device="cuda")
        N.gs_render_fwd(tr.proj[0], tr.n, tr.vals[0], tr.ranges[0], bc[0], tr.bg, img, Tf, nc, wk)
        K = 8
        T = ((W + 15) // 16) * ((H + 15) // 16)
        tcost = torch.empty(T, dtype=torch.int64, device="cuda")
        cum = torch.empty(T, dtype=torch.int64, device="cuda")
        bounds = torch.empty(K + 1, dtype=torch.int64, device="cuda")
        order = torch.empty(B, dtype=torch.int32, device="cuda")
        score = torch.empty(B, dtype=torch.float32, device="cuda")
        reps = 20
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        N.gs_tile_split(wk[2], W, H, K, tcost, cum, bounds)
        a.record()
        for _ in range(reps):
            N.gs_tile_split(wk[2], W, H, K, tcost, cum, bounds)
        b.record()
        torch.cuda.synchronize()
        split_us = a.elapsed_time(b) / reps * 1e3
        a.record()
        for _ in range(reps):
            N.gs_view_order(tr.jaccard, B, 1, order, score)
        b.record()
        torch.cuda.synchronize()
        order_us = a.elapsed_time(b) / reps * 1e3
        bl = bounds.cpu().tolist()
        tc = tcost.cpu()
        parts = [int(tc[bl[k]:bl[k + 1]].sum()) for k in range(K)]
        mean = max(1.0, sum(parts) / K)
        schedule = {"tile_split": {"parts": K, "tiles": T, "us": round(split_us, 2),
                                   "max_part_over_mean": round(max(parts) / mean, 4),
                                   "cost": "entries each pixel's warp walked (gs_render_fwd work[2]), one view"},
                    "view_order": {"views": B, "unit": 1, "us": round(order_us, 2),
                                   "order": order.cpu().tolist()}}
    except Exception as e:  # reported, never fatal to the benchmark line
        schedule = {"error": str(e)[:200]}
    # opacity pruning of the trained state into scratch outputs (the trainer is left as is):
    # count pass, then the timed compaction of parameters and both moments
    try:
        n = tr.n
        min_opacity = 0.005
        min_logit = math.log(min_opacity / (1.0 - min_opacity))
        ws_p = torch.empty(max(N.gs_prune_workspace_size(n), 256), dtype=torch.uint8, device="cuda")
        nk = torch.zeros(1, dtype=torch.int64, device="cuda")
        sets = [tr.params, tr.exp_avg, tr.exp_avg_sq]
        k = N.gs_prune(sets, n, min_logit, None, 0, ws_p, nk, sync=True)
        free, _ = torch.cuda.mem_get_info()
        if 3 * 240 * max(k, 1) > free // 2:
            raise RuntimeError("not enough free device memory for the pruning outputs")
        outs = [torch.empty((15, max(k, 1), 4), dtype=torch.float32, device="cuda") for _ in sets]
        reps = 10
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        N.gs_prune(sets, n, min_logit, outs, max(k, 1), ws_p, nk)
        a.record()
        for _ in range(reps):
            N.gs_prune(sets, n, min_logit, outs, max(k, 1), ws_p, nk)
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) / reps * 1e3
        # algorithmic bytes: every Gaussian's opacity logit read twice (count and scatter
        # passes, 4 B each) and, per kept Gaussian, 3 x 240 B read and written
        nbytes = 2 * 4 * n + k * 3 * 240 * 2
        del outs
        prune = {"min_opacity": min_opacity, "kept": k, "of": n, "us": round(us, 2),
                 "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
    except Exception as e:
        prune = {"error": str(e)[:200]}
    schedule = dict(schedule or {})
    schedule["prune"] = prune

    # projected footprints of one view (the GPU's radii): the fraction below 2 % of the image
    # width, the property the large workloads are drawn to have
    rad = tr.proj[0][1, :, 3].contiguous().view(torch.int32)
    vis_r = rad[rad > 0].float()
    footprint = {"view": batch_of(0)[0][0], "visible": int(vis_r.numel()),
                 "frac_radius_below_2pct_width": round(float((vis_r < 0.02 * cfg.width).float().mean()), 5)
                 if vis_r.numel() else None,
                 "radius_p90_px": float(torch.quantile(vis_r[:1 << 24], 0.9)) if vis_r.numel() else None}
    sm_count = torch.cuda.get_device_properties(local).multi_processor_count
    FP32_PEAK_TFLOPS = fp32_peak_tflops(sm_count, max_sm_mhz(local))
    fp32_src = f"derived: {sm_count} SM x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x the maximum SM clock"
    avg = {k: sum(v) / len(v) for k, v in per_call.items()}
    share = {k: sum(v) / total_ms for k, v in per_call.items()}
    peak_hbm, hbm_src = hbm_peak()
    flops = {"render_fwd": FWD_FLOPS_PER_PAIR * ev, "render_bwd": BWD_FLOPS_PER_PAIR * ev,
             "loss": LOSS_FLOPS_PER_PIXEL * cfg.width * cfg.height}
    work_note = (f"per launch: {ev:.4g} pixel-Gaussian pairs evaluated through termination "
                 f"({used:.4g} accumulated, {walked:.4g} walked back; the forward's warps evaluated "
                 f"{warp_pairs:.4g}); fwd {FWD_FLOPS_PER_PAIR}, bwd {BWD_FLOPS_PER_PAIR} flops per evaluated pair")
    # dominant single kernel: the entry points that launch one kernel (gs_bin_sort_batch launches several)
    single = [k for k in ("render_bwd", "render_fwd", "project", "project_bwd", "sparse_adam", "project_bwd_adam")
              if k in per_call]
    dominant = max(single, key=lambda k: sum(per_call[k]))
    roof = {}
    if dominant in flops:
        ach = flops[dominant] / (avg[dominant] / 1e3) / 1e12
        roof = {"kernel": "k_" + dominant, "bound": "alu", "achieved": ach, "peak": FP32_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": ach / FP32_PEAK_TFLOPS, "traffic": measured_traffic(dominant, cfg.name),
                "peak_source": fp32_src,
                "measured_peak": fp32_meas, "frac_of_measured": ach / fp32_meas if fp32_meas else None,
                "measured_peak_source": "gs_probe_ffma in this run: 8 FFMA chains per thread, full occupancy",
                "work": work_note}
    else:
        roof = {"kernel": "k_" + dominant, "bound": "hbm", "achieved": None, "peak": peak_hbm, "unit": "GB/s",
                "frac": None, "traffic": measured_traffic(dominant, cfg.name), "peak_source": hbm_src}
    others = {}
    for k in ("render_fwd", "render_bwd", "loss"):
        if k in flops and k in avg:
            ach = flops[k] / (avg[k] / 1e3) / 1e12
            others[k] = {"bound": "alu", "achieved_tflops": round(ach, 3), "frac": round(ach / FP32_PEAK_TFLOPS, 4),
                         "frac_of_measured": round(ach / fp32_meas, 4) if fp32_meas else None}
    if "project_bwd_adam" in avg:
        # algorithmic bytes: every view's visibility bitset (one bit per Gaussian, the trainer
        # hands over gs_visible_sets' bitsets) and its visible Gaussians' screen-space
        # gradients (48 B); for the updated Gaussians, the parameters (240 B) and moments
        # (480 B) read once and all three written (720 B)
        nu = int(tr.n_union.item())
        offs = tr.offsets.cpu().tolist()
        vis = sum(offs[b + 1] - offs[b] for b in range(cfg.batch))
        nbytes = cfg.batch * ((tr.n + 31) // 32) * 4 + vis * 48 + nu * (240 + 480 + 720)
        gbs = nbytes / (avg["project_bwd_adam"] / 1e3) / 1e9
        others["project_bwd_adam"] = {"bound": "hbm", "achieved_gbs": round(gbs, 1),
                                      "frac": round(gbs / peak_hbm, 4), "bytes": nbytes, "peak_source": hbm_src}

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        log("end to end")
        host_t = torch.empty((cfg.n_views, 3, cfg.height, cfg.width), dtype=torch.float32).pin_memory()
        host_t.copy_(targets)  # device -> pinned host, no pageable temporary

        def host_batch(ids):
            # a batch of consecutive views is a slice of the pinned array (itself pinned);
            # otherwise one pinned gather per distinct batch, made before the timed steps
            if ids == list(range(ids[0], ids[0] + len(ids))):
                return host_t[ids[0]:ids[0] + len(ids)]
            key = tuple(ids)
            if key not in gathered:
                gathered[key] = host_t[list(ids)].pin_memory()
            return gathered[key]

        gathered = {}
        for s in range(args.steps):
            host_batch(batch_of(args.warmup + s)[0])
        for s in range(2):
            ids, bc = batch_of(s)
            tr.step(bc, host_batch(ids))
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for s in range(args.steps):
            ids, bc = batch_of(args.warmup + s)
            tr.step(bc, host_batch(ids))
        torch.cuda.synchronize()
        t_e2e = time.perf_counter() - t0
        t_e2e = max_over_ranks(t_e2e, dist, "cuda")
        del host_t, gathered
        e2e = {"value": views / t_e2e, "unit": UNIT,
               "h2d_bytes_per_step": cfg.batch * 3 * cfg.height * cfg.width * 4,
               "d2h_bytes_per_step": 4 + cfg.batch * 16}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        log("CPU baseline: calibrating")
        smp = OracleSampler(args.config, P=P, cams=cams, jit=jit)
        smp.calibrate(10.0)
        log(f"CPU baseline: bands of {smp.rows} rows; starting the processes")
        smp.start()
        log(f"CPU baseline: {smp.workers} processes; one round")
        v, wall, views = smp.round()
        smp.stop()
        cpu = {"value": v, "unit": UNIT, "cores": smp.workers, "kind": "oracle",
               "sample": f"one round ({views:.3f} views): " + smp.describe(wall)}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {**workload, "l2": "flushed between timed steps (512 MB write)",
                           "parallelism": "replicas" if world > 1 else "single"},
                "roofline": roof,
                "kernels": {"ms_avg": {k: round(v, 4) for k, v in avg.items()},
                            "calls": "project, bin_sort, visible_sets and project_bwd_adam once per batch, the rest once per view",
                            "share": {k: round(v, 4) for k, v in share.items()}, **others},
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "schedule": schedule,
                "footprint": footprint, "work_counts": f"one orbit: {orbit} batches, every view once",
                "clocks": clk.summary(), "instances_per_view": int(st[:, 0].float().mean().item())}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
