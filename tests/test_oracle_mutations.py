"""The oracle's pins bite: each plausible mistake, planted in a copy of the oracle's source on
the CPU, makes at least one pin fail.

Every mutation names a text that occurs exactly once in oracle.cpp and its replacement; the
copy is compiled into a temporary directory and the oracle's pin files run against it in a
child process (``GS_ORACLE_LIB`` points the wrapper at the copy).  The child must fail.  The
copies are built and checked concurrently, one child per host core.  Nothing here touches the
oracle the other tests use.

The mistakes cover every stage: the projection and its backward, compositing forward and
backward, the loss, the batch-scaled Adam, the visible sets, the binning sort, pruning,
densification, the balanced tile split and the view order.  Dropping the compositing step's
skip of a positive exponent is not among them: every conic the projection produces is
positive definite (the 0.3 dilation), so its exponent is never positive and that change
alters no output.
"""
import concurrent.futures
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")
PIN_FILES = ["test_oracle_edges.py", "test_oracle_projection.py", "test_oracle_densify.py", "test_oracle_pins.py",
             "test_oracle_next.py"]

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

    # backward: sign of the screen position's depth derivative
    "bwd_u_depth_sign": ("dpc[2] += -du * k.fx * x / (z * z) - dv * k.fy * y / (z * z);",
                         "dpc[2] += du * k.fx * x / (z * z) - dv * k.fy * y / (z * z);"),
    # backward: d conic_A / d a with c in place of c^2
    "bwd_conic_ga": ("const double ga = dconic[0] * (-c * c / d2)", "const double ga = dconic[0] * (-c / d2)"),
    # backward: sign of a term of d conic_B / d b
    "bwd_conic_gb": ("dconic[1] * (-1.0 / det - 2 * b * b / d2)", "dconic[1] * (-1.0 / det + 2 * b * b / d2)"),
    # backward: the shared off-diagonal's gradient not split between the two entries
    "bwd_offdiag_not_halved": ("const double G2[2][2] = {{ga, 0.5 * gb}, {0.5 * gb, gc}};",
                               "const double G2[2][2] = {{ga, gb}, {gb, gc}};"),
    # backward: d(T Sig T^T) / dT without its factor 2
    "bwd_dTm_factor": ("acc += 2.0 * G2[ii][jj] * p.Tm[jj][m] * p.Sig[m][l];",
                       "acc += G2[ii][jj] * p.Tm[jj][m] * p.Sig[m][l];"),
    # backward: d(fx / z) / dz as -fx / z
    "bwd_J00_depth": ("dpc[2] += dJ[0][0] * (-k.fx / (z * z)) + dJ[1][1] * (-k.fy / (z * z));",
                      "dpc[2] += dJ[0][0] * (-k.fx / z) + dJ[1][1] * (-k.fy / (z * z));"),
    # backward: d(-fx x / z^2) / dz without its factor 2
    "bwd_J02_depth_factor": ("dpc[2] += dJ[0][2] * (2.0 * k.fx * x / (z * z * z));",
                             "dpc[2] += dJ[0][2] * (k.fx * x / (z * z * z));"),
    # backward: the y clamp's branches exchanged
    "bwd_clamp_y_branches": ("if (p.cly) {", "if (!p.cly) {"),
    # backward: d(M M^T) / dM not symmetrised
    "bwd_sigma_not_symmetrised": ("acc += (dSig[l][n2] + dSig[n2][l]) * M[n2][m];", "acc += dSig[l][n2] * M[n2][m];"),
    # backward: log-scale gradient without ds / dlog s = s
    "bwd_scale_chain": ("dls[m] = acc * p.s[m];", "dls[m] = acc;"),
    # backward: a sign in d R / d w
    "bwd_quat_w_sign": ("dq[0] = 2 * (-qz * dRq[0][1]", "dq[0] = 2 * (qz * dRq[0][1]"),
    # backward: the quaternion's normalisation left out of its gradient
    "bwd_quat_no_normalisation": ("dqraw[l] = (dq[l] - p.qn[l] * dot) / p.qlen;", "dqraw[l] = dq[l] / p.qlen;"),
    # backward: a colour channel clamped at 0 still passes gradients
    "bwd_colour_mask": ("if (p.raw[ch] < 0) continue;", "(void)0;"),
    # backward: sigmoid derivative without (1 - o)
    "bwd_dlogit": ("const double dlogit = dopac * p.o * (1.0 - p.o);", "const double dlogit = dopac * p.o;"),
    # backward: SH gradient written to the coefficient index instead of the (k, channel) float
    "bwd_sh_layout": ("G(3 + f / 4, f % 4) += gch * p.Y[kk];", "G(3 + kk / 4, kk % 4) += gch * p.Y[kk];"),
    # compositing: sign of the exponent's cross term
    "power_cross_sign": ("const double power = -0.5 * (A * dx * dx + Cc * dy * dy) - B * dx * dy;",
                         "const double power = -0.5 * (A * dx * dx + Cc * dy * dy) + B * dx * dy;"),
    # compositing: pixel corner instead of pixel centre
    "pixel_corner": ("const double dx = (px + 0.5) - in.uvzo[4 * g + 0];", "const double dx = px - in.uvzo[4 * g + 0];"),
    # compositing: alpha capped at 0.999
    "alpha_cap": ("const float a_min = 1.0f / 255.0f, a_max = 0.99f, t_min = 1e-4f;",
                  "const float a_min = 1.0f / 255.0f, a_max = 0.999f, t_min = 1e-4f;"),
    # compositing: no skip of alphas below 1/255
    "no_alpha_skip": ("if (f32(alpha) < a_min) continue;", "if (f32(alpha) <= 0.0f) continue;"),
    # compositing: termination tested on the transmittance before the Gaussian
    "termination_before": ("if (f32(Tn) < t_min) {  // stop before this Gaussian",
                           "if (f32(pr.T) < t_min) {  // stop before this Gaussian"),
    # work counts: the entry that ends the walk not counted as evaluated
    "count_eval_terminator": ("pr.n_eval = j - start + 1;", "pr.n_eval = j - start;"),
    # work counts: list positions counted as accumulated entries
    "count_used_positions": ("++pr.n_used;", "pr.n_used = pr.n_contrib;"),
    # compositing: colour weighted by the transmittance after the Gaussian
    "weight_after": ("pr.C[c] += in.rgb[3 * g + c] * alpha * pr.T;", "pr.C[c] += in.rgb[3 * g + c] * alpha * Tn;"),
    # compositing: the background not attenuated by the final transmittance
    "background_unattenuated": ("img[c * P + pix] = pr.C[c] + pr.T * bg[c];", "img[c * P + pix] = pr.C[c] + bg[c];"),
    # compositing backward: the colour behind a Gaussian not divided by (1 - alpha)
    "bwd_no_one_minus_alpha": ("dalpha += (u.T * col[c] - after[c] / (1.0 - u.alpha)) * dC[c];",
                               "dalpha += (u.T * col[c] - after[c]) * dC[c];"),
    # compositing backward: the background left out of the light behind the Gaussians
    "bwd_suffix_no_background": ("double after[3] = {pr.T * bg[0], pr.T * bg[1], pr.T * bg[2]};",
                                 "double after[3] = {0, 0, 0};"),
    # compositing backward: a capped alpha still passes gradients to opacity and the conic
    "bwd_capped_alpha_gradient": ("if (u.clamped) continue;", "(void)u.clamped;"),
    # compositing backward: the cross term's derivative halved
    "bwd_cross_half": ("g2d[9 * g + 3] += dpow * (-u.dx * u.dy);", "g2d[9 * g + 3] += dpow * (-0.5 * u.dx * u.dy);"),
    # compositing backward: sign of the screen-position gradient
    "bwd_du_sign": ("g2d[9 * g + 0] += dpow * (A * u.dx + B * u.dy);", "g2d[9 * g + 0] -= dpow * (A * u.dx + B * u.dy);"),
    # compositing backward: the v gradient with the offsets swapped
    "bwd_dv_swapped": ("g2d[9 * g + 1] += dpow * (B * u.dx + Cc * u.dy);", "g2d[9 * g + 1] += dpow * (B * u.dy + Cc * u.dx);"),
    # compositing backward: opacity gradient without the Gaussian's falloff
    "bwd_opacity_no_falloff": ("g2d[9 * g + 5] += dalpha * u.G;", "g2d[9 * g + 5] += dalpha;"),
    # compositing backward: colour gradient without the transmittance
    "bwd_colour_no_T": ("g2d[9 * g + 6 + c] += u.alpha * u.T * dC[c];", "g2d[9 * g + 6 + c] += u.alpha * dC[c];"),
    # loss: C2 not squared
    "loss_C2": ("const double C1 = 0.01 * 0.01, C2 = 0.03 * 0.03;", "const double C1 = 0.01 * 0.01, C2 = 0.03;"),
    # loss: window with sigma^2 = 1.5
    "loss_sigma": ("h[k] = std::exp(-((k - 5) * (k - 5)) / (2.0 * 1.5 * 1.5));",
                   "h[k] = std::exp(-((k - 5) * (k - 5)) / (2.0 * 1.5));"),
    # loss: window not normalised
    "loss_window_unnormalised": ("for (int k = 0; k < 11; ++k) h[k] /= s;", "(void)s;"),
    # loss: covariance without the product of the means
    "loss_covariance": ("sxy = exy[p] - ux * uy;", "sxy = exy[p];"),
    # loss: replicated edges instead of zero padding
    "loss_edge_replicate": ("if (yy < 0 || yy >= H) continue;", "yy = std::min(std::max(yy, 0), H - 1);"),
    # loss gradient: sign of the E[x^2] partial
    "loss_dexx_sign": ("dexx[p] = -S / B2;", "dexx[p] = S / B2;"),
    # loss gradient: SSIM term added instead of subtracted
    "loss_ssim_gradient_sign": ("dimg[c * P + p] = scale * (w_l1 * sg / n - w_ssim * dssim);",
                                "dimg[c * P + p] = scale * (w_l1 * sg / n + w_ssim * dssim);"),
    # loss gradient: d E[x^2] / dx taken as x
    "loss_square_derivative": ("const double dssim = (t1[p] + 2 * X[p] * t2[p] + Yt[p] * t3[p]) / n;",
                               "const double dssim = (t1[p] + X[p] * t2[p] + Yt[p] * t3[p]) / n;"),
    # Adam: learning rate scaled by b instead of sqrt(b)
    "adam_lr_linear": ("const double lr_b = lr * std::sqrt((double)batch);", "const double lr_b = lr * (double)batch;"),
    # Adam: beta1 not raised to the batch size
    "adam_beta1_unscaled": ("const double b1 = std::pow(beta1, batch), b2 = std::pow(beta2, batch);",
                            "const double b1 = beta1, b2 = std::pow(beta2, batch);"),
    # Adam: no bias correction of the second moment
    "adam_no_bias_correction": ("bc2 = 1.0 - std::pow(b2, (double)step);", "bc2 = 1.0;"),
    # Adam: epsilon inside the square root
    "adam_eps_inside_sqrt": ("p[e] -= lr_b * mh / (std::sqrt(vh) + eps);", "p[e] -= lr_b * mh / std::sqrt(vh + eps);"),
    # Adam: second moment of |g| instead of g^2
    "adam_v_not_squared": ("v[e] = b2 * v[e] + (1.0 - b2) * g * g;", "v[e] = b2 * v[e] + (1.0 - b2) * std::fabs(g);"),
    # Adam: gradient not cleared after the update
    "adam_gradient_kept": ("gr[e] = 0.0;", "(void)0;"),
    # step: the update set taken from the first view only
    "step_union_first_view": ("for (int b = 0; b < B && !any; ++b) any = radii[(size_t)b * N + i] > 0;",
                              "any = radii[i] > 0;"),
    # step: per-view losses summed, not averaged
    "step_loss_sum": ("loss += loss_one(img.data(), targets + (int64_t)b * 3 * P, W, H, w_l1, w_ssim, 1.0 / B, dimg.data());",
                      "loss += loss_one(img.data(), targets + (int64_t)b * 3 * P, W, H, w_l1, w_ssim, 1.0, dimg.data());"),
    # visible sets: union size without the intersection subtracted
    "jaccard_union": ("const int64_t un = (int64_t)sets[i].size() + (int64_t)sets[j].size() - n;",
                      "const int64_t un = (int64_t)sets[i].size() + (int64_t)sets[j].size();"),
    # visible sets: weight 1 for an empty union
    "jaccard_empty_union": ("jac[i * B + j] = un == 0 ? 0.0f :", "jac[i * B + j] = un == 0 ? 1.0f :"),
    # visible sets: radius 0 counted as visible in the union
    "union_radius_zero": ("for (int b = 0; b < B && !any; ++b) any = radius[(int64_t)b * N + i] > 0;",
                          "for (int b = 0; b < B && !any; ++b) any = radius[(int64_t)b * N + i] >= 0;"),
    # binning: a tile's range ends one entry early
    "range_end": ("ranges[2 * t + 1] = (uint32_t)(j + 1);", "ranges[2 * t + 1] = (uint32_t)j;"),
    # binning: unstable sort
    "unstable_sort": ("std::stable_sort(inst.begin(), inst.end(),", "std::sort(inst.begin(), inst.end(),"),
    # binning: depth key not the fp32 depth
    "depth_key": ("float zf = f32(uvzo[4 * i + 2]);", "float zf = f32(uvzo[4 * i + 2] * 1.0000001);"),
    # tile split: a block ending on a target moves to the next part
    "split_left": ("if ((unsigned __int128)K * cum[i] <= (unsigned __int128)k * total) ++c;",
                   "if ((unsigned __int128)K * cum[i] < (unsigned __int128)k * total) ++c;"),
    # tile split: exclusive cumulative sum
    "split_exclusive_cum": ("run += tile_cost[i];\n    cum[i] = run;", "cum[i] = run;\n    run += tile_cost[i];"),
    # view order: the largest score first
    "order_max": ("if (best < 0 || s < best_s) {", "if (best < 0 || s > best_s) {"),
    # view order: ties to the higher index
    "order_tie_high": ("if (best < 0 || s < best_s) {", "if (best < 0 || s <= best_s) {"),
    # view order: scores against every earlier unit, not the previous one
    "order_all_previous": ("prev = cur;", "prev.insert(prev.end(), cur.begin(), cur.end());"),
    # pruning: a logit equal to the threshold dropped
    "prune_strict": ("if (!(logit >= min_logit)) continue;", "if (!(logit > min_logit)) continue;"),
    # pruning: the opacity read from the wrong lane
    "prune_lane": ("const float logit = planes[0][(0 * n + i) * 4 + 3];", "const float logit = planes[0][(0 * n + i) * 4 + 2];"),
    # densification statistic: L1 length of the screen gradient
    "stat_l1_length": ("stat[2 * i + 0] += std::sqrt(du * du + dv * dv);", "stat[2 * i + 0] += std::fabs(du) + std::fabs(dv);"),
}


def _compile(src_text, out_dir):
    path = os.path.join(out_dir, "oracle_mut.cpp")
    with open(path, "w") as fh:
        fh.write(src_text)
    lib = os.path.join(out_dir, "liboracle_mut.so")
    subprocess.run(["g++", "-O1", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    "-o", lib, path], check=True)
    return lib


def _run_pins(src_text):
    """Builds the given source and runs the pin files against it; returns (exit code, output)."""
    with tempfile.TemporaryDirectory() as d:
        lib = _compile(src_text, d)
        env = dict(os.environ, GS_ORACLE_LIB=lib)
        cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + \
              [os.path.join(ROOT, "tests", f) for f in PIN_FILES]
        r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-3000:] + r.stderr[-1000:]


@pytest.fixture(scope="module")
def outcomes():
    """Every mutant (and the unmutated copy, key None) run concurrently; futures by name."""
    text = open(SRC).read()
    pool = concurrent.futures.ThreadPoolExecutor(max_workers=max(2, os.cpu_count() or 2))
    futs = {None: pool.submit(_run_pins, text)}
    for name, (old, new) in MUTATIONS.items():
        if text.count(old) == 1:
            futs[name] = pool.submit(_run_pins, text.replace(old, new))
    yield futs
    pool.shutdown(wait=True)


def test_mutation_targets_occur_once():
    text = open(SRC).read()
    for name, (old, _) in MUTATIONS.items():
        assert text.count(old) == 1, name


def test_unmutated_copy_passes_the_same_pins(outcomes):
    rc, out = outcomes[None].result()
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(outcomes, name):
    assert name in outcomes, f"mutation {name}: target text not found once"
    rc, out = outcomes[name].result()
    assert rc != 0, f"mutation {name} passed every pin:\n{out}"
    assert "failed" in out, out
