"""Host-side helpers of the GPU parity tests (tests/parity.py), on the CPU: the conversions
between the oracle's arrays and the library's documented layouts, and the tolerance rule."""
import numpy as np

import parity


def test_projection_planes_round_trip_the_documented_layout():
    # proj [3][N][4]: q0 = (u, v, z, opacity), q1 = (A, B, C, radius as int32 bits),
    # q2 = (r, g, b, tiles as int32 bits); a culled Gaussian (radius 0) is all zero
    pr = dict(uvzo=np.array([[10.5, 20.25, 3.0, 0.5], [1.0, 2.0, 3.0, 0.7]]),
              conic=np.array([[0.1, -0.02, 0.3], [0.4, 0.5, 0.6]]),
              radius=np.array([7, 0], np.int32),
              rgb=np.array([[0.2, 0.4, 0.6], [0.9, 0.9, 0.9]]),
              tiles=np.array([4, 0], np.int32))
    P = parity.proj_planes_from_oracle(pr)
    assert P.shape == (3, 2, 4) and P.dtype == np.float32
    assert P[1, 0, 3:].view(np.int32)[0] == 7 and P[2, 0, 3:].view(np.int32)[0] == 4
    assert (P[:, 1] == 0).all()
    uvzo, conic, radius, rgb = parity.oracle_inputs_from_planes(P)
    assert np.array_equal(uvzo[0], pr["uvzo"][0]) and np.array_equal(conic[0], pr["conic"][0].astype(np.float32))
    assert radius.tolist() == [7, 0]
    assert np.array_equal(rgb[0], pr["rgb"][0].astype(np.float32))


def test_grad2d_record_maps_to_the_oracle_order():
    # gs_render_bwd's record [n][12]: (du, dv, dopacity, 0, dA, dB, dC, 0, dr, dg, db, 0);
    # the oracle's n x 9: (du, dv, dA, dB, dC, dopacity, dr, dg, db)
    rec = np.array([[1, 2, 3, 0, 4, 5, 6, 0, 7, 8, 9, 0]], np.float64)
    assert parity.grad2d_oracle_layout(rec).tolist() == [[1, 2, 4, 5, 6, 3, 7, 8, 9]]


def test_gradient_tolerance_rule():
    ref = np.array([1.0, 1e-3, 0.0, -2.0])
    ok = ref * (1 + 0.9e-3) + np.array([0.0, 0.0, 0.9e-6, 0.0])
    assert not parity.allclose_grad(ok, ref).any()
    bad = ref * (1 + 1.2e-3) + np.array([0.0, 0.0, 1.2e-6, 0.0])
    assert parity.allclose_grad(bad, ref)[[0, 2, 3]].all()


def test_flagged_pixel_bound():
    # one flipped decision moves a pixel by at most ~1e-2 of the largest colour (a late stop)
    b = parity.flag_img_bound(np.array([[0.5, 1.0, 0.25]]), bg=(0.0, 0.0, 2.0))
    assert abs(b - ((1e-2 * (1 + parity.MARGIN) + 1e-4) * 2.0 + parity.IMG_ATOL)) < 1e-15
