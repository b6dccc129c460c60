"""The projection and densification pins bite: each plausible mistake, planted in a copy of the oracle's source
on the CPU, makes at least one pin fail.

Every mutation names a text that occurs exactly once in oracle.cpp and its replacement; the
copy is compiled into a temporary directory and the pins of ``test_oracle_projection.py``,
``test_oracle_densify.py`` and ``test_oracle_pins.py`` run against it in a child process
(``GS_ORACLE_LIB`` points the wrapper at the copy).  The child must fail.  Nothing here
touches the oracle the other tests use.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

MUTATIONS = {
    # R(q) transposed: Sigma = R^T S^2 R
    "transposed_rotation": ("acc += Rq[i][l] * p.s[l] * p.s[l] * Rq[j][l];",
                            "acc += Rq[l][i] * p.s[l] * p.s[l] * Rq[l][j];"),
    # sign of the off-axis Jacobian term of the u row
    "j02_sign": ("p.J[0][2] = -k.fx * p.xr / z;", "p.J[0][2] = k.fx * p.xr / z;"),
    # the v row's off-axis term takes the x ratio
    "j12_wrong_ratio": ("p.J[1][2] = -k.fy * p.yr / z;", "p.J[1][2] = -k.fy * p.xr / z;"),
    # camera rotation transposed in T = J W
    "camera_rotation_transposed": ("acc += p.J[i][l] * k.R[l][j];", "acc += p.J[i][l] * k.R[j][l];"),
    # SH view direction from the mean to the camera
    "sh_direction_reversed": ("p.dir[i] = g.mu[i] - cam[i];", "p.dir[i] = cam[i] - g.mu[i];"),
    # no field-of-view clamp of x/z in the Jacobian
    "no_clamp_x": ("p.xr = std::min(std::max(p.xr, -limx), limx);", "(void)limx;"),
    # clamp limit without the 1.3 factor
    "clamp_factor": ("const double limx = 1.3 * (0.5 * k.W / k.fx)", "const double limx = 1.0 * (0.5 * k.W / k.fx)"),
    # screen position with the principal point of the other axis
    "u_principal_point": ("p.u = k.fx * x / z + k.cx;", "p.u = k.fx * x / z + k.cy;"),
    # scale squared dropped in Sigma (S instead of S S^T)
    "scale_not_squared": ("acc += Rq[i][l] * p.s[l] * p.s[l] * Rq[j][l];", "acc += Rq[i][l] * p.s[l] * Rq[j][l];"),
    # the low-pass dilation dropped on the off-diagonal side: b gets 0.3 instead of c
    "dilation_on_b": ("p.b = p.cov[0][1];", "p.b = p.cov[0][1] + 0.3;"),
    # wrong sign of an l = 1 basis function
    "sh_l1_sign": ("set(2, c1 * z, 0, 0, c1);", "set(2, -c1 * z, 0, 0, -c1);"),
    # backward: camera rotation not transposed when pulling the camera-space gradient back
    "bwd_camera_rotation": ("for (int l = 0; l < 3; ++l) dmu[j] += k.R[l][j] * dpc[l];",
                            "for (int l = 0; l < 3; ++l) dmu[j] += k.R[j][l] * dpc[l];"),
    # backward: wrong sign in the clamped branch of the Jacobian's depth derivative
    "bwd_clamp_branch_sign": ("dpc[2] += dJ[0][2] * (k.fx * p.xr / (z * z));",
                              "dpc[2] -= dJ[0][2] * (k.fx * p.xr / (z * z));"),
    # backward: view-direction gradient with the wrong sign
    "bwd_sh_direction_sign": ("dmu[l] += (dd[l] - p.d[l] * ddot) / p.dlen;",
                              "dmu[l] -= (dd[l] - p.d[l] * ddot) / p.dlen;"),
    # densification: split offset along the transposed rotation
    "split_rotation_transposed": ("off += R[r][j] * s[j] * (double)normals[6 * i + 3 * child + j];",
                                  "off += R[j][r] * s[j] * (double)normals[6 * i + 3 * child + j];"),
    # densification: children scaled up instead of down
    "split_scale_sign": ("for (int j = 0; j < 3; ++j) c[1][j] = p[1][j] - std::log(1.6);",
                         "for (int j = 0; j < 3; ++j) c[1][j] = p[1][j] + std::log(1.6);"),
    # densification: a mean exactly at the threshold not selected
    "densify_threshold_strict": ("if (!(avg >= grad_threshold)) continue;", "if (!(avg > grad_threshold)) continue;"),
}


def _compile(src_text, out_dir):
    path = os.path.join(out_dir, "oracle_mut.cpp")
    with open(path, "w") as fh:
        fh.write(src_text)
    lib = os.path.join(out_dir, "liboracle_mut.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", lib, path], check=True)
    return lib


def _run_pins(lib):
    env = dict(os.environ, GS_ORACLE_LIB=lib)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_oracle_projection.py"),
           os.path.join(ROOT, "tests", "test_oracle_densify.py"),
           os.path.join(ROOT, "tests", "test_oracle_pins.py") + "::test_single_isotropic_gaussian_closed_form"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_mutation_targets_occur_once():
    text = open(SRC).read()
    for name, (old, _) in MUTATIONS.items():
        assert text.count(old) == 1, name


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_projection_pins_catch_planted_mistake(name):
    old, new = MUTATIONS[name]
    text = open(SRC).read()
    assert text.count(old) == 1
    with tempfile.TemporaryDirectory() as d:
        lib = _compile(text.replace(old, new), d)
        r = _run_pins(lib)
    assert r.returncode != 0, f"mutation {name} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]


def test_unmutated_copy_passes_the_same_pins():
    with tempfile.TemporaryDirectory() as d:
        lib = _compile(open(SRC).read(), d)
        r = _run_pins(lib)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
