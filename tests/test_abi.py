"""Host-side checks of the C ABI (no GPU needed): every symbol include/gs.h declares is
exported by libgs.so, and argument errors are rejected on the host before any CUDA call."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gs.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gs_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gaussian_splatting_gb300 import build
    build.build()
    from gaussian_splatting_gb300 import _native
    return _native.load()


def test_header_declares_the_eight_step_calls():
    names = declared_functions()
    for f in ["gs_project", "gs_bin_sort", "gs_render_fwd", "gs_loss", "gs_render_bwd", "gs_project_bwd",
              "gs_sparse_adam", "gs_visible_sets"]:
        assert f in names


def test_library_exports_every_declared_symbol(lib):
    from gaussian_splatting_gb300 import _native
    names = declared_functions()
    assert set(names) == set(_native.EXPORTS)
    for name in names:
        assert hasattr(lib, name), name


def test_host_side_argument_errors(lib):
    from gaussian_splatting_gb300 import _native as N
    import scenes
    cam = N.camera(scenes.make_cameras(0)[0])
    assert lib.gs_version() >= 1
    # negative n / NULL pointers / bad sizes fail on the host with GS_ERR_INVALID
    assert lib.gs_project(None, -1, C.byref(cam), None, None) == N.GS_ERR_INVALID
    assert b"bad n" in lib.gs_last_error()
    assert lib.gs_project(None, 5, C.byref(cam), None, None) == N.GS_ERR_INVALID
    assert lib.gs_loss(None, None, 0, 4, 0.8, 0.2, 1.0, None, 0, None, None, 0, None) == N.GS_ERR_INVALID
    assert lib.gs_visible_sets(None, 0, 10, None, 0, None, None, None, None, None, None, None, 0,
                               None) == N.GS_ERR_INVALID
    # the batched projection: a bitset stride below ceil(n / 32)
    assert lib.gs_project_batch(None, 100, C.byref(cam), 1, None, None, 0, None) == N.GS_ERR_INVALID
    assert lib.gs_sparse_adam(None, None, None, None, 10, None, None, 10, 1e-3, 0.9, 0.999, 1e-15, 0, 1, None, 0,
                              None) == N.GS_ERR_INVALID
    bad = N.camera(scenes.make_cameras(0)[0])
    bad.width = 0
    assert lib.gs_render_fwd(None, 0, None, None, C.byref(bad), None, None, None, None, None, None, None,
                             None) == N.GS_ERR_INVALID
    # the tile launch order: n_tiles out of range, NULL pointers (no cost source, no output)
    assert lib.gs_tile_order(None, None, -1, 4, 4, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_order(None, None, 4, 65536, 4, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_order(None, None, 4, 4, 0, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_order(None, None, 4, 4, 9, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_order(None, None, 10, 3, 4, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_order(None, None, 0, 7, 4, None, None) == N.GS_OK
    # misaligned workspace / capacity bounds for the sort
    assert lib.gs_bin_sort(None, 0, C.byref(cam), 8, 10, None, None, 1 << 30, 64, 64, None, None) == N.GS_ERR_INVALID
    # the scheduling helpers: parts, batch and unit out of range, NULL pointers
    assert lib.gs_tile_split(None, 64, 64, 0, None, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_split(None, 64, 64, 1025, None, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_tile_split(None, 64, 64, 4, None, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_view_order(None, 65, 1, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_view_order(None, 4, 5, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_view_order(None, 4, 1, None, None, None) == N.GS_ERR_INVALID
    # pruning: set count out of range, NULL output with a nonzero stride
    assert lib.gs_prune(None, 0, 10, C.c_float(0.0), None, 0, None, 0, None, None, None) == N.GS_ERR_INVALID
    assert lib.gs_prune(None, 5, 10, C.c_float(0.0), None, 0, None, 0, None, None, None) == N.GS_ERR_INVALID
    # the batched sort: batch < 1, NULL pointer arrays
    assert lib.gs_bin_sort_batch(None, 0, 0, C.byref(cam), 256, 10, None, None, 0, None, 64, None, None) \
        == N.GS_ERR_INVALID
    assert lib.gs_bin_sort_batch(None, 1, 0, C.byref(cam), 256, 10, None, None, 0, None, 64, None, None) \
        == N.GS_ERR_INVALID


def test_workspace_sizes_are_pure_host_functions(lib):
    from gaussian_splatting_gb300 import _native as N
    import scenes
    cam = scenes.make_cameras(1)[0]
    a = N.gs_bin_sort_workspace_size(300_000, 10_000_000, cam)
    b = N.gs_bin_sort_workspace_size(300_000, 20_000_000, cam)
    assert 0 < a < b
    # a batch holds depth buffers for up to 8 views and capacity-sized tile-sort buffers for the
    # views that share a tile-sort launch (as many as fit 1 GiB): one set at 100M instances...
    big = [N.gs_bin_sort_batch_workspace_size(b, 300_000, 100_000_000, [cam] * b) for b in (1, 4, 8, 16)]
    assert big[0] == N.gs_bin_sort_workspace_size(300_000, 100_000_000, cam)
    assert (big[1] - big[0]) * 7 == (big[2] - big[0]) * 3 and big[2] == big[3]  # equal per-view depth parts
    # ... six sets at 10M (160 MB each), so a batch of 4 holds four and one of 8 or 16 six
    b = [N.gs_bin_sort_batch_workspace_size(k, 300_000, 10_000_000, [cam] * k) for k in (1, 4, 8, 16)]
    assert b[0] == a and b[2] == b[3]
    assert b[1] - b[0] == 3 * b[0]  # four views: four depth parts and four tile sets
    assert N.gs_loss_workspace_size(1236, 820) > 0
    assert N.gs_visible_sets_workspace_size(4, 300_000) > 0
    assert N.gs_visible_sets_workspace_size(65, 10) == 0


def test_launch_count_bookkeeping():
    import scenes
    from gaussian_splatting_gb300.trainer import bin_sort_launches
    # every radix pass of a sort runs inside one cooperative launch; per group of up to 8 views
    # one zeroing, one depth-sort and one publishing launch, and the tile sorts of as many views
    # per launch as have ping-pong buffers within 1 GiB (six at 10M instances, one at 100M)
    assert bin_sort_launches(1, 10_000_000) == 4
    assert bin_sort_launches(4, 10_000_000) == 4
    assert bin_sort_launches(4, 100_000_000) == 7
    assert bin_sort_launches(16, 10_000_000) == 2 * (3 + 2)
    assert bin_sort_launches(16, 100_000_000) == 22
