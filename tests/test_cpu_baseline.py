"""The CPU baseline's sampling (bench.py's OracleSampler), on the host.

The Gaussians the sampler hands a process must be all that its band of rows needs: the band's
camera renders the same image from them alone as from the whole scene.  The bands must sit
where the sampler says: one in the middle of each equal share of the view's rows, aligned to
the 16-row tiles.
"""
import numpy as np

import bench
import oracle
import scenes


def test_band_gaussians_are_all_the_band_needs():
    smp = bench.OracleSampler(0, workers=8)
    smp.rows = 16
    cfg = smp.cfg
    rows_seen = []
    for k in range(8):
        cam, rows, idx = smp._band_idx(k)
        r0 = int(round(smp.cams[0].cy - cam.cy))
        assert 0 < idx.size < smp.P.shape[1]
        band = oracle.render_view(smp.P[:, idx], cam)
        whole = oracle.render_view(smp.P, cam)
        assert np.array_equal(band, whole), k
        assert band.any()
        # the band's camera differs from the view's only by its principal point and height
        assert cam.width == smp.cams[0].width and cam.height == rows == 16
        assert cam.fx == smp.cams[0].fx and cam.fy == smp.cams[0].fy
        rows_seen.extend(range(r0, r0 + rows))
    assert sorted(rows_seen) == list(range(cfg.height))  # eight bands of 16 rows tile the view


def test_band_positions_are_stratum_middles():
    cfg = scenes.CONFIGS[4]
    P = np.zeros((15, 8, 4), np.float32)
    P[0, :, 2] = np.linspace(-1.0, 1.0, 8)
    cams = scenes.make_cameras(4)
    H = cfg.height
    for workers in (1, 3, 4, 16):
        smp = bench.OracleSampler(4, P=P, cams=cams, jit=P, workers=workers)
        smp.rows = 16
        starts = []
        for k in range(workers):
            cam, rows, _ = smp._band_idx(k)
            r0 = int(round(cams[0].cy - cam.cy)) if k < min(H // 16, workers) else None
            if r0 is None:
                continue
            assert rows == 16 and r0 % 16 == 0 and 0 <= r0 <= H - 16
            mid = (2 * k + 1) * H // (2 * workers)
            assert r0 <= mid < r0 + 32, (workers, k, r0, mid)
            starts.append(r0)
        assert starts == sorted(set(starts))
    one = bench.OracleSampler(4, P=P, cams=cams, jit=P, workers=1)
    one.rows = 16
    cam, _, _ = one._band_idx(0)
    assert abs((cams[0].cy - cam.cy) - H / 2) <= 16  # a lone band sits at mid-height, not at the top
