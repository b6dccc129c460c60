"""The allocation-free loss entry point (gs_loss_noalloc) against the workspace one (gs_loss).

gs_loss_noalloc exists for callers that cannot hand the library device memory -- memory
owned by another allocator under a fixed budget, or code that must not call cudaMalloc /
cudaFree because they can synchronise the device.  It keeps its partial sums in a fixed
array inside libgs.so.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover - CPU container
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gaussian_splatting_gb300 import _native as N  # noqa: E402

from parity import RTOL  # noqa: E402

pytestmark = pytest.mark.gpu


def _pair(H, W, seed):
    rng = np.random.default_rng(seed)
    x = rng.uniform(0, 1, size=(3, H, W)).astype(np.float32)
    y = np.clip(x + rng.normal(0, 0.1, size=x.shape), 0, 1).astype(np.float32)
    return torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda()


def _with_workspace(x, y, H, W, scale, acc_start):
    ws_b = N.gs_loss_workspace_size(W, H)
    ws = torch.empty(ws_b, dtype=torch.uint8, device="cuda")
    loss = torch.full((1,), acc_start, dtype=torch.float32, device="cuda")
    d = torch.zeros((3, H, W), dtype=torch.float32, device="cuda")
    N.gs_loss(x, y, W, H, 0.8, 0.2, scale, loss, acc_start != 0.0, d, ws, ws_b)
    torch.cuda.synchronize()
    return float(loss.item()), d.cpu().numpy()


def _without(x, y, H, W, scale, acc_start):
    loss = torch.full((1,), acc_start, dtype=torch.float32, device="cuda")
    d = torch.zeros((3, H, W), dtype=torch.float32, device="cuda")
    N.gs_loss_noalloc(x, y, W, H, 0.8, 0.2, scale, loss, acc_start != 0.0, d)
    torch.cuda.synchronize()
    return float(loss.item()), d.cpu().numpy()


def test_noalloc_loss_matches_workspace_loss_on_two_calls_in_a_row():
    # two consecutive calls (different sizes, the second accumulating): the shared array
    # keeps the first call's contents, which must not leak into the second
    for H, W, scale, acc in [(820, 1236, 0.25, 0.0), (131, 77, 1.0, 0.5)]:
        x, y = _pair(H, W, H + W)
        l_ref, d_ref = _with_workspace(x, y, H, W, scale, acc)
        l_new, d_new = _without(x, y, H, W, scale, acc)
        assert l_new == pytest.approx(l_ref, rel=1e-6)
        tol = RTOL * np.abs(d_ref) + 1e-6 * np.abs(d_ref).max()
        assert (np.abs(d_new - d_ref) <= tol).all()


def test_noalloc_loss_rejects_images_beyond_its_scratch():
    # 8192 x 8192 needs 256 * 256 * 3 = 196,608 partial sums > 65,536
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    big = torch.zeros((3, 8192, 8192), dtype=torch.float32, device="cuda")
    with pytest.raises(N.GSError) as e:
        N.gs_loss_noalloc(big, big, 8192, 8192, 0.8, 0.2, 1.0, loss, False, big)
    assert e.value.status == N.GS_ERR_INVALID
    assert "scratch" in str(e.value)
