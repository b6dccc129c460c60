"""Register use and spills of every kernel, as ptxas reports them for the library's own build
flags (``nvcc -Xptxas -v``, cross-compiled for sm_103a; no GPU needed).

The hot kernels are sized to a register budget (64 per thread for the sorts, the compositing
and the batched projection, so that four or more CTAs fit an SM); a change that makes one
spill more than the bytes recorded here, or use more registers than its budget, fails.
"""
import concurrent.futures
import os
import re
import shutil
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from gaussian_splatting_gb300 import build as B  # noqa: E402

# kernel -> (registers at most, spill store bytes at most, spill load bytes at most)
BUDGET = {
    "k_tile_sort": (64, 24, 76),
    "k_depth_sort": (64, 4, 16),
    "k_depth_sort_wide": (64, 0, 0),
    "k_render_fwd": (64, 0, 0),
    "k_render_bwd": (64, 0, 0),
    "k_project_fwd_batch": (64, 0, 0),
    "k_project_fwd": (64, 0, 0),
    "k_project_bwd_adam": (128, 0, 0),
    "k_project_bwd": (128, 0, 0),
    "k_loss_fused": (80, 0, 0),
    "k_sparse_adam": (64, 0, 0),
}


def _ptxas_report():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out_dir = tempfile.mkdtemp()

    def one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        r = subprocess.run([nvcc, *B.NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o", obj], capture_output=True,
                           text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        return r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2)) as ex:
        reports = list(ex.map(one, B.sources()))
    shutil.rmtree(out_dir, ignore_errors=True)
    stats = {}
    for text in reports:
        _parse(text, stats)
    return stats


def _parse(text, stats):
    """Each entry function's registers and spill bytes, from the per-function blocks of one
    file's report (the -warn-spills warnings at its top name no kernel and are skipped)."""
    name = None
    for line in text.splitlines():
        if "warning" in line:
            continue
        m = re.search(r"(?:Compiling entry function|Function properties for) '?([^' ]+)'?", line)
        if m:
            k = re.findall(r"\d+(k_[A-Za-z0-9_]+?)(?:ILb[01]E|E)", m.group(1))
            name = k[0] if k else None
            continue
        if name is None:
            continue
        rec = stats.setdefault(name, [0, 0, 0])
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            rec[1] = max(rec[1], int(m.group(1)))
            rec[2] = max(rec[2], int(m.group(2)))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            rec[0] = max(rec[0], int(m.group(1)))


def test_kernels_stay_within_their_register_and_spill_budgets():
    stats = _ptxas_report()
    missing = [k for k in BUDGET if k not in stats]
    assert not missing, f"kernels not found in the ptxas report: {missing}"
    over = {k: (stats[k], BUDGET[k]) for k in BUDGET
            if any(s > b for s, b in zip(stats[k], BUDGET[k]))}
    assert not over, f"(registers, spill stores, spill loads) above budget: {over}"
    # every other kernel spills nothing
    spilling = {k: v for k, v in stats.items() if k not in BUDGET and (v[1] or v[2])}
    assert not spilling, spilling
