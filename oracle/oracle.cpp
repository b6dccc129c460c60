// Oracle for the 3D Gaussian Splatting training step -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, double-precision CPU restatement of one training step, written
// as straight loops in the order the method takes its steps.  Only the tests,
// the package smoke check and the benchmark's CPU-baseline leg may load it; the
// product path never does.  It shares no code, header, table or constant with
// the CUDA path.
//
// Sources for the method (web pages on distributed 3DGS training):
//  * Grendel-GS notes, "背景知识" (parameter table: position 3, scale 3, quaternion 4,
//    opacity 1, SH 48) and "训练流程" (transform -> render by depth-sorted alpha
//    compositing -> L1+SSIM loss -> backpropagation -> update);
//  * Grendel-GS notes §1.2 (16x16 pixel tiles), §4.2 (sqrt(batch) learning rate,
//    beta^batch momentum);
//  * Odin summary, "研究背景与动机" (a view renders, backpropagates and updates only
//    the primitives it sees) and §1 (Jaccard weight, 0 for an empty union).
// The pages give the outline only.  The remaining constants (EWA low-pass 0.3,
// J clamp 1.3 tan(fov/2), 3-sigma radius, alpha clamp 0.99 and skip below
// 1/255, termination below T = 1e-4, SH basis and sign convention, SSIM
// window / constants / zero padding, Adam bias correction) are the readings
// the tests pin; each function below names the step it restates.
//
// Discrete decisions (culls, radius ceiling, tile rectangle, alpha skip,
// termination) are taken on fp32-rounded operands against fp32 thresholds,
// the precision the kernels decide in.  Each function can report a per-element
// "margin": the smallest relative distance of any decision operand from its
// threshold, so that a test can set aside the rare element whose decision an
// ulp-level difference could flip.
//
// Parity pins (see tests/test_oracle_*.py): closed form of one isotropic
// Gaussian; anisotropic, rotated, off-axis Gaussians against scipy's quaternion
// rotation, a numpy covariance product and a finite-difference Jacobian of the
// pinhole map; hand-worked closed forms off the axis, for quarter turns and
// beyond the field-of-view clamp; the view-dependent colour from two opposite
// cameras; SH against scipy's complex harmonics and by quadrature, brute-force
// per-pixel compositing (image, transmittance and the walk's work counts),
// compositing invariants, central finite differences of
// the whole forward (also from an oblique camera with a clamped Gaussian), SSIM
// identities, Adam closed form at t = 1, set identities, balanced splits of known
// cost profiles, worked view orders on block-structured weights; closed forms of
// one opaque Gaussian over a coloured background (forward and backward, the 0.99
// cap), equal depth keys in the binning sort, Adam with a large epsilon and the
// update set of a two-view step.  A mutation test plants mistakes in copies of
// this file, in every stage, and checks that the pins fail.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

constexpr int TILE = 16;
constexpr double PI = 3.14159265358979323846;

// ---------------------------------------------------------------- camera
struct Cam {
  double R[3][3];  // world -> camera rows
  double t[3];
  double fx, fy, cx, cy, znear;
  int W, H, Tx, Ty;
};

Cam load_cam(const double* c, int W, int H) {
  Cam k;
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) k.R[i][j] = c[3 * i + j];
  for (int i = 0; i < 3; ++i) k.t[i] = c[9 + i];
  k.fx = c[12]; k.fy = c[13]; k.cx = c[14]; k.cy = c[15]; k.znear = c[16];
  k.W = W; k.H = H;
  k.Tx = (W + TILE - 1) / TILE;
  k.Ty = (H + TILE - 1) / TILE;
  return k;
}

// ---------------------------------------------------------------- parameters
// Parameter planes [15][N][4]: p0 = (mean, opacity logit), p1 = (log scale, 0),
// p2 = quaternion (w, x, y, z), p3..p14 = sh[k][c] flattened as 3k + c.
struct Gauss {
  double mu[3], ls[3], q[4], logit, sh[16][3];
};

inline double P(const double* params, int64_t N, int plane, int64_t i, int lane) {
  return params[((int64_t)plane * N + i) * 4 + lane];
}

Gauss load_gauss(const double* params, int64_t N, int64_t i) {
  Gauss g;
  for (int k = 0; k < 3; ++k) g.mu[k] = P(params, N, 0, i, k);
  g.logit = P(params, N, 0, i, 3);
  for (int k = 0; k < 3; ++k) g.ls[k] = P(params, N, 1, i, k);
  for (int k = 0; k < 4; ++k) g.q[k] = P(params, N, 2, i, k);
  for (int f = 0; f < 48; ++f) g.sh[f / 3][f % 3] = P(params, N, 3 + f / 4, i, f % 4);
  return g;
}

// ---------------------------------------------------------------- SH basis
// Real spherical harmonics up to degree 3, k = l*l + l + m.  Real form of the
// complex Y_l^m with the Condon-Shortley phase: sqrt2*Re(Y_l^m) for m > 0,
// sqrt2*Im(Y_l^|m|) for m < 0, Y_l^0 for m = 0.  Written as polynomials of the
// unit direction (x, y, z); dY holds their partial derivatives.
void sh_basis(const double d[3], double Y[16], double dY[16][3]) {
  const double x = d[0], y = d[1], z = d[2];
  const double c0 = 0.5 * std::sqrt(1.0 / PI);
  const double c1 = std::sqrt(3.0 / (4.0 * PI));
  const double a = 0.5 * std::sqrt(15.0 / PI);
  const double b = 0.25 * std::sqrt(5.0 / PI);
  const double c = 0.25 * std::sqrt(15.0 / PI);
  const double e = 0.25 * std::sqrt(35.0 / (2.0 * PI));
  const double f = 0.5 * std::sqrt(105.0 / PI);
  const double g = 0.25 * std::sqrt(21.0 / (2.0 * PI));
  const double h = 0.25 * std::sqrt(7.0 / PI);
  const double i = 0.25 * std::sqrt(105.0 / PI);
  auto set = [&](int k, double v, double gx, double gy, double gz) {
    Y[k] = v; dY[k][0] = gx; dY[k][1] = gy; dY[k][2] = gz;
  };
  set(0, c0, 0, 0, 0);
  set(1, -c1 * y, 0, -c1, 0);
  set(2, c1 * z, 0, 0, c1);
  set(3, -c1 * x, -c1, 0, 0);
  set(4, a * x * y, a * y, a * x, 0);
  set(5, -a * y * z, 0, -a * z, -a * y);
  set(6, b * (2 * z * z - x * x - y * y), -2 * b * x, -2 * b * y, 4 * b * z);
  set(7, -a * x * z, -a * z, 0, -a * x);
  set(8, c * (x * x - y * y), 2 * c * x, -2 * c * y, 0);
  set(9, -e * y * (3 * x * x - y * y), -6 * e * x * y, -e * (3 * x * x - 3 * y * y), 0);
  set(10, f * x * y * z, f * y * z, f * x * z, f * x * y);
  set(11, -g * y * (4 * z * z - x * x - y * y), 2 * g * x * y, -g * (4 * z * z - x * x - 3 * y * y),
      -8 * g * y * z);
  set(12, h * z * (2 * z * z - 3 * x * x - 3 * y * y), -6 * h * x * z, -6 * h * y * z,
      h * (6 * z * z - 3 * x * x - 3 * y * y));
  set(13, -g * x * (4 * z * z - x * x - y * y), -g * (4 * z * z - 3 * x * x - y * y), 2 * g * x * y,
      -8 * g * x * z);
  set(14, i * z * (x * x - y * y), 2 * i * x * z, -2 * i * y * z, i * (x * x - y * y));
  set(15, -e * x * (x * x - 3 * y * y), -e * (3 * x * x - 3 * y * y), 6 * e * x * y, 0);
}

// ---------------------------------------------------------------- decisions
inline float f32(double v) { return (float)v; }
inline double relm(double v, double thr) {  // relative distance of v from thr
  return std::fabs(v - thr) / std::max(std::fabs(thr), 1e-30);
}
inline int64_t floordiv(int64_t a, int64_t b) {
  int64_t q = a / b;
  if ((a % b != 0) && ((a < 0) != (b < 0))) --q;
  return q;
}

// ---------------------------------------------------------------- projection
// "Transform" step (Grendel-GS notes, 训练流程): 3D Gaussian -> screen position,
// depth, footprint radius and colour.
struct Proj {
  bool vis = false;
  double pc[3] = {0, 0, 0};
  double s[3], o, qn[4], qlen, Rq[3][3], Sig[3][3];
  double xr, yr;          // clamped x/z and y/z used in J
  bool clx, cly;          // clamp active
  double J[2][3], Tm[2][3], cov[2][2];
  double a, b, c, det, conic[3];
  double u = 0, v = 0, z = 0;
  int r = 0;
  int rect[4] = {0, 0, 0, 0};
  int tiles = 0;
  double dir[3], dlen, d[3], Y[16], dY[16][3], raw[3], rgb[3] = {0, 0, 0};
  double margin = 1e30;   // nearest decision that can change an output (see project_one)
  double rmargin = 1e30;  // the integer radius and tile rectangle values (0: either may differ)
};

void rect_of(double u, double v, int r, const Cam& k, int rect[4]) {
  // Tile rectangle of the radius-r square around (u, v): tiles [x0, x1) x [y0, y1).
  // Integer form of clamp(floor((u -+ r)/16)), exact for any float u.
  double uc = std::min(std::max(u, -1e9), 1e9), vc = std::min(std::max(v, -1e9), 1e9);
  int64_t fu = (int64_t)std::floor((double)f32(uc)), fv = (int64_t)std::floor((double)f32(vc));
  int64_t x0 = floordiv(fu - r, TILE), x1 = floordiv(fu + r, TILE) + 1;
  int64_t y0 = floordiv(fv - r, TILE), y1 = floordiv(fv + r, TILE) + 1;
  rect[0] = (int)std::min<int64_t>(std::max<int64_t>(x0, 0), k.Tx);
  rect[1] = (int)std::min<int64_t>(std::max<int64_t>(y0, 0), k.Ty);
  rect[2] = (int)std::min<int64_t>(std::max<int64_t>(x1, 0), k.Tx);
  rect[3] = (int)std::min<int64_t>(std::max<int64_t>(y1, 0), k.Ty);
}

// Relative margin below which a discrete decision counts as undecided (the parity tests'
// threshold; the kernels' fp32 operands carry relative errors of a few 1e-6).
constexpr double kDecisionMargin = 1e-5;

// Would the tile rectangle `alt` instead of `rect` change any output?  Only through the tiles
// in one and not the other, and there only at a pixel where the Gaussian passes the
// compositing skip tests (power <= 0, alpha >= 1/255), both taken with the decision margin so
// that a pixel on the edge of the skip counts.  The Gaussian's conic, opacity and screen
// position must be set in p.
bool reaches(const Proj& p, const Gauss& g, const Cam& k, const int rect[4], const int alt[4]) {
  (void)g;
  if (std::memcmp(rect, alt, 4 * sizeof(int)) == 0) return false;
  const int x0 = std::min(rect[0], alt[0]), x1 = std::max(rect[2], alt[2]);
  const int y0 = std::min(rect[1], alt[1]), y1 = std::max(rect[3], alt[3]);
  auto in = [](const int r[4], int tx, int ty) { return tx >= r[0] && tx < r[2] && ty >= r[1] && ty < r[3]; };
  const double a_min = (double)(1.0f / 255.0f) * (1.0 - kDecisionMargin);
  for (int ty = y0; ty < y1; ++ty)
    for (int tx = x0; tx < x1; ++tx) {
      if (in(rect, tx, ty) == in(alt, tx, ty)) continue;
      for (int py = ty * TILE; py < std::min(ty * TILE + TILE, k.H); ++py)
        for (int px = tx * TILE; px < std::min(tx * TILE + TILE, k.W); ++px) {
          const double dx = (px + 0.5) - p.u, dy = (py + 0.5) - p.v;
          const double power = -0.5 * (p.conic[0] * dx * dx + p.conic[2] * dy * dy) - p.conic[1] * dx * dy;
          if (power > kDecisionMargin) continue;
          if (std::min(0.99, p.o * std::exp(power)) >= a_min) return true;
        }
    }
  return false;
}

Proj project_one(const Gauss& g, const Cam& k) {
  Proj p;
  for (int i = 0; i < 3; ++i)
    p.pc[i] = k.R[i][0] * g.mu[0] + k.R[i][1] * g.mu[1] + k.R[i][2] * g.mu[2] + k.t[i];
  const double x = p.pc[0], y = p.pc[1], z = p.pc[2];
  p.margin = std::min(p.margin, relm(z, k.znear));
  if (f32(z) <= f32(k.znear)) return p;  // behind the near plane

  for (int i = 0; i < 3; ++i) p.s[i] = std::exp(g.ls[i]);
  p.o = 1.0 / (1.0 + std::exp(-g.logit));
  p.qlen = std::sqrt(g.q[0] * g.q[0] + g.q[1] * g.q[1] + g.q[2] * g.q[2] + g.q[3] * g.q[3]);
  for (int i = 0; i < 4; ++i) p.qn[i] = g.q[i] / p.qlen;
  const double w = p.qn[0], qx = p.qn[1], qy = p.qn[2], qz = p.qn[3];
  double Rq[3][3] = {
      {1 - 2 * (qy * qy + qz * qz), 2 * (qx * qy - w * qz), 2 * (qx * qz + w * qy)},
      {2 * (qx * qy + w * qz), 1 - 2 * (qx * qx + qz * qz), 2 * (qy * qz - w * qx)},
      {2 * (qx * qz - w * qy), 2 * (qy * qz + w * qx), 1 - 2 * (qx * qx + qy * qy)}};
  std::memcpy(p.Rq, Rq, sizeof(Rq));
  // Sigma = R S S^T R^T, S = diag(s)
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j) {
      double acc = 0;
      for (int l = 0; l < 3; ++l) acc += Rq[i][l] * p.s[l] * p.s[l] * Rq[j][l];
      p.Sig[i][j] = acc;
    }
  // EWA: J of the perspective map at the (clamped) camera-space point
  const double limx = 1.3 * (0.5 * k.W / k.fx), limy = 1.3 * (0.5 * k.H / k.fy);
  p.xr = x / z; p.yr = y / z;
  p.clx = p.xr < -limx || p.xr > limx;
  p.cly = p.yr < -limy || p.yr > limy;
  p.xr = std::min(std::max(p.xr, -limx), limx);
  p.yr = std::min(std::max(p.yr, -limy), limy);
  p.J[0][0] = k.fx / z; p.J[0][1] = 0; p.J[0][2] = -k.fx * p.xr / z;
  p.J[1][0] = 0; p.J[1][1] = k.fy / z; p.J[1][2] = -k.fy * p.yr / z;
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 3; ++j) {
      double acc = 0;
      for (int l = 0; l < 3; ++l) acc += p.J[i][l] * k.R[l][j];
      p.Tm[i][j] = acc;
    }
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 2; ++j) {
      double acc = 0;
      for (int l = 0; l < 3; ++l)
        for (int m = 0; m < 3; ++m) acc += p.Tm[i][l] * p.Sig[l][m] * p.Tm[j][m];
      p.cov[i][j] = acc;
    }
  p.a = p.cov[0][0] + 0.3;  // low-pass dilation of one pixel-variance 0.3
  p.b = p.cov[0][1];
  p.c = p.cov[1][1] + 0.3;
  p.det = p.a * p.c - p.b * p.b;
  p.margin = std::min(p.margin, p.det / (p.a * p.c));
  if (f32(p.det) <= 0.0f) return p;
  p.conic[0] = p.c / p.det;
  p.conic[1] = -p.b / p.det;
  p.conic[2] = p.a / p.det;
  // radius: 3 sigma of the larger eigenvalue, rounded up
  const double mid = 0.5 * (p.a + p.c);
  const double lam = mid + std::sqrt(std::max(mid * mid - p.det, 0.0));
  const double r3 = 3.0 * std::sqrt(lam);
  const double rfr = r3 - std::floor(r3);
  p.rmargin = std::min(rfr, 1.0 - rfr) / r3;
  p.r = (int)std::ceil(f32(r3));
  p.u = k.fx * x / z + k.cx;
  p.v = k.fy * y / z + k.cy;
  p.z = z;
  rect_of(p.u, p.v, p.r, k, p.rect);
  // The radius reaches the rest of the step only through the tile rectangle: a ceiling within
  // the margin counts as a decision if the neighbouring radius gives a rectangle that adds or
  // drops a tile where the Gaussian has a pixel with alpha >= 1/255 (see reaches()).
  if (p.rmargin < kDecisionMargin) {
    int alt[4];
    rect_of(p.u, p.v, rfr < 0.5 ? p.r - 1 : p.r + 1, k, alt);
    if (reaches(p, g, k, p.rect, alt)) p.margin = std::min(p.margin, p.rmargin);
  }
  {  // could a floor(u) or floor(v) one step away give another rectangle?  The kernels round
     // u = fx x / z + cx in fp32; |u_fp32 - u| stays within 1e-6 (|u - cx| (1 + cond_x +
     // cond_z) + |cx|), cond_i = (sum_j |R_ij mu_j| + |t_i|) / |p_i| being the condition
     // number of the camera-space coordinate (four times the roundings of the fma chain,
     // the division, the scaling and the offset), so only a screen position that close to an
     // integer can be floored differently.
    double cond[3];
    for (int i = 0; i < 3; ++i) {
      const double terms = std::fabs(k.R[i][0] * g.mu[0]) + std::fabs(k.R[i][1] * g.mu[1]) +
                           std::fabs(k.R[i][2] * g.mu[2]) + std::fabs(k.t[i]);
      cond[i] = terms / std::max(std::fabs(p.pc[i]), 1e-30);
    }
    for (int ax = 0; ax < 2; ++ax) {
      double q = ax == 0 ? p.u : p.v;
      const double c0 = ax == 0 ? k.cx : k.cy;
      double fr = q - std::floor(q);
      double eps = 1e-6 * (std::fabs(q - c0) * (1.0 + cond[ax] + cond[2]) + std::fabs(c0));
      if (fr < eps || fr > 1.0 - eps) {
        int alt[4];
        double q2 = fr < eps ? q - 0.5 : q + 0.5;
        rect_of(ax == 0 ? q2 : p.u, ax == 0 ? p.v : q2, p.r, k, alt);
        if (std::memcmp(alt, p.rect, sizeof(alt)) != 0) p.rmargin = 0.0;
        if (reaches(p, g, k, p.rect, alt)) p.margin = 0.0;
      }
    }
  }
  if (p.rect[0] >= p.rect[2] || p.rect[1] >= p.rect[3]) { p.r = 0; return p; }
  p.tiles = (p.rect[2] - p.rect[0]) * (p.rect[3] - p.rect[1]);
  // view-dependent colour from degree-3 SH, +0.5, clamped at 0
  double cam[3];
  for (int i = 0; i < 3; ++i) cam[i] = -(k.R[0][i] * k.t[0] + k.R[1][i] * k.t[1] + k.R[2][i] * k.t[2]);
  for (int i = 0; i < 3; ++i) p.dir[i] = g.mu[i] - cam[i];
  p.dlen = std::sqrt(p.dir[0] * p.dir[0] + p.dir[1] * p.dir[1] + p.dir[2] * p.dir[2]);
  for (int i = 0; i < 3; ++i) p.d[i] = p.dir[i] / p.dlen;
  sh_basis(p.d, p.Y, p.dY);
  for (int ch = 0; ch < 3; ++ch) {
    double acc = 0;
    for (int kk = 0; kk < 16; ++kk) acc += g.sh[kk][ch] * p.Y[kk];
    p.raw[ch] = acc + 0.5;
    p.rgb[ch] = std::max(p.raw[ch], 0.0);
  }
  p.vis = true;
  return p;
}

// ---------------------------------------------------------------- compositing
// "Render" step: per pixel, the Gaussians of its tile in depth order,
// front-to-back alpha compositing.  One record per evaluated Gaussian.
struct Contrib {
  int64_t g;       // Gaussian index
  double alpha;    // after the 0.99 clamp
  double T;        // transmittance before this Gaussian
  double G;        // exp(power)
  bool clamped;    // o*G > 0.99
  double dx, dy;
};

struct PixelResult {
  double C[3];
  double T;
  uint32_t n_contrib;
  uint32_t n_eval;  // list entries evaluated: through the terminating one, else the whole list
  uint32_t n_used;  // list entries accumulated
  double margin;
  std::vector<Contrib> used;
};

struct View2D {  // per-Gaussian screen-space inputs of the compositing step
  const double* uvzo;   // N x 4 (u, v, z, opacity)
  const double* conic;  // N x 3 (A, B, C)
  const double* rgb;    // N x 3
};

PixelResult composite_pixel(const View2D& in, const uint32_t* vals, uint32_t start, uint32_t end,
                            int px, int py, bool keep) {
  PixelResult pr;
  pr.C[0] = pr.C[1] = pr.C[2] = 0;
  pr.T = 1.0;
  pr.n_contrib = 0;
  pr.n_eval = end - start;
  pr.n_used = 0;
  pr.margin = 1e30;
  const float a_min = 1.0f / 255.0f, a_max = 0.99f, t_min = 1e-4f;
  for (uint32_t j = start; j < end; ++j) {
    const int64_t g = vals[j];
    const double dx = (px + 0.5) - in.uvzo[4 * g + 0];
    const double dy = (py + 0.5) - in.uvzo[4 * g + 1];
    const double A = in.conic[3 * g + 0], B = in.conic[3 * g + 1], Cc = in.conic[3 * g + 2];
    const double power = -0.5 * (A * dx * dx + Cc * dy * dy) - B * dx * dy;
    pr.margin = std::min(pr.margin, std::fabs(power) / 1e-4);
    if (f32(power) > 0.0f) continue;
    const double G = std::exp(power);
    const double oa = in.uvzo[4 * g + 3] * G;
    const bool clamped = f32(oa) > a_max;
    const double alpha = clamped ? (double)a_max : oa;
    pr.margin = std::min(pr.margin, relm(oa, a_max));
    pr.margin = std::min(pr.margin, relm(oa, a_min));
    if (f32(alpha) < a_min) continue;
    const double Tn = pr.T * (1.0 - alpha);
    pr.margin = std::min(pr.margin, relm(Tn, t_min));
    if (f32(Tn) < t_min) {  // stop before this Gaussian
      pr.n_eval = j - start + 1;
      break;
    }
    for (int c = 0; c < 3; ++c) pr.C[c] += in.rgb[3 * g + c] * alpha * pr.T;
    if (keep) pr.used.push_back({g, alpha, pr.T, G, clamped, dx, dy});
    pr.T = Tn;
    pr.n_contrib = j - start + 1;
    ++pr.n_used;
  }
  return pr;
}

// ---------------------------------------------------------------- loss
// "Loss" step: L1 + SSIM (Grendel-GS notes, 训练流程).  Weights 0.8 / 0.2,
// 11x11 Gaussian window with sigma 1.5 (normalised to sum 1), zero padding,
// C1 = 0.01^2, C2 = 0.03^2.  Direct 2-D window sums.
void window11(double w[11][11]) {
  double h[11], s = 0;
  for (int k = 0; k < 11; ++k) { h[k] = std::exp(-((k - 5) * (k - 5)) / (2.0 * 1.5 * 1.5)); s += h[k]; }
  for (int k = 0; k < 11; ++k) h[k] /= s;
  for (int i = 0; i < 11; ++i)
    for (int j = 0; j < 11; ++j) w[i][j] = h[i] * h[j];
}

// out[p] = sum_{i,j} w[i][j] * in[p + (i-5, j-5)], zero outside the image
void conv11(const double* in, double* out, int W, int H, const double w[11][11]) {
  for (int y = 0; y < H; ++y)
    for (int x = 0; x < W; ++x) {
      double acc = 0;
      for (int i = 0; i < 11; ++i) {
        int yy = y + i - 5;
        if (yy < 0 || yy >= H) continue;
        for (int j = 0; j < 11; ++j) {
          int xx = x + j - 5;
          if (xx < 0 || xx >= W) continue;
          acc += w[i][j] * in[(int64_t)yy * W + xx];
        }
      }
      out[(int64_t)y * W + x] = acc;
    }
}

double loss_one(const double* img, const double* tgt, int W, int H, double w_l1, double w_ssim,
                double scale, double* dimg /* may be null */) {
  const int64_t P = (int64_t)W * H;
  const double n = 3.0 * (double)P;
  const double C1 = 0.01 * 0.01, C2 = 0.03 * 0.03;
  double w[11][11];
  window11(w);
  double l1 = 0, ssim = 0;
  std::vector<double> x2(P), y2(P), xy(P), mx(P), my(P), exx(P), eyy(P), exy(P);
  std::vector<double> dmx(P), dexx(P), dexy(P), t1(P), t2(P), t3(P);
  for (int c = 0; c < 3; ++c) {
    const double* X = img + c * P;
    const double* Yt = tgt + c * P;
    for (int64_t p = 0; p < P; ++p) {
      x2[p] = X[p] * X[p]; y2[p] = Yt[p] * Yt[p]; xy[p] = X[p] * Yt[p];
      l1 += std::fabs(X[p] - Yt[p]);
    }
    conv11(X, mx.data(), W, H, w);
    conv11(Yt, my.data(), W, H, w);
    conv11(x2.data(), exx.data(), W, H, w);
    conv11(y2.data(), eyy.data(), W, H, w);
    conv11(xy.data(), exy.data(), W, H, w);
    for (int64_t p = 0; p < P; ++p) {
      const double ux = mx[p], uy = my[p];
      const double sxx = exx[p] - ux * ux, syy = eyy[p] - uy * uy, sxy = exy[p] - ux * uy;
      const double A1 = 2 * ux * uy + C1, A2 = 2 * sxy + C2;
      const double B1 = ux * ux + uy * uy + C1, B2 = sxx + syy + C2;
      const double S = (A1 * A2) / (B1 * B2);
      ssim += S;
      // partials of S(mu_x, E[x^2], E[xy]) at fixed target statistics
      dmx[p] = (2 * uy * (A2 - A1)) / (B1 * B2) - 2 * ux * S * (1.0 / B1 - 1.0 / B2);
      dexx[p] = -S / B2;
      dexy[p] = 2 * A1 / (B1 * B2);
    }
    if (dimg) {
      // adjoint of the zero-padded symmetric window sum is the same window sum
      conv11(dmx.data(), t1.data(), W, H, w);
      conv11(dexx.data(), t2.data(), W, H, w);
      conv11(dexy.data(), t3.data(), W, H, w);
      for (int64_t p = 0; p < P; ++p) {
        const double diff = X[p] - Yt[p];
        const double sg = diff > 0 ? 1.0 : (diff < 0 ? -1.0 : 0.0);
        const double dssim = (t1[p] + 2 * X[p] * t2[p] + Yt[p] * t3[p]) / n;
        dimg[c * P + p] = scale * (w_l1 * sg / n - w_ssim * dssim);
      }
    }
  }
  return scale * (w_l1 * (l1 / n) + w_ssim * (1.0 - ssim / n));
}

// ---------------------------------------------------------------- project backward
// Reverse mode of project_one: screen-space gradients -> parameter gradients.
// gout: planes [15][N][4] accumulated with +=.
void project_bwd_one(const Gauss& g, const Proj& p, const Cam& k, const double du, const double dv,
                     const double dconic[3], const double dopac, const double drgb[3], double* gout,
                     int64_t N, int64_t i) {
  if (!p.vis) return;
  auto G = [&](int plane, int lane) -> double& { return gout[((int64_t)plane * N + i) * 4 + lane]; };
  double dpc[3] = {0, 0, 0};
  double dmu[3] = {0, 0, 0};
  const double x = p.pc[0], y = p.pc[1], z = p.pc[2];
  // u = fx x / z + cx, v = fy y / z + cy
  dpc[0] += du * k.fx / z;
  dpc[1] += dv * k.fy / z;
  dpc[2] += -du * k.fx * x / (z * z) - dv * k.fy * y / (z * z);
  // conic = (c, -b, a) / det of the dilated 2D covariance (a, b, c)
  const double a = p.a, b = p.b, c = p.c, det = p.det, d2 = det * det;
  const double ga = dconic[0] * (-c * c / d2) + dconic[1] * (b * c / d2) + dconic[2] * (-b * b / d2);
  const double gb = dconic[0] * (2 * b * c / d2) + dconic[1] * (-1.0 / det - 2 * b * b / d2) +
                    dconic[2] * (2 * a * b / d2);
  const double gc = dconic[0] * (-b * b / d2) + dconic[1] * (a * b / d2) + dconic[2] * (-a * a / d2);
  // cov = Tm Sig Tm^T ; b is the shared off-diagonal entry
  const double G2[2][2] = {{ga, 0.5 * gb}, {0.5 * gb, gc}};
  double dSig[3][3], dTm[2][3];
  for (int l = 0; l < 3; ++l)
    for (int m = 0; m < 3; ++m) {
      double acc = 0;
      for (int ii = 0; ii < 2; ++ii)
        for (int jj = 0; jj < 2; ++jj) acc += p.Tm[ii][l] * G2[ii][jj] * p.Tm[jj][m];
      dSig[l][m] = acc;
    }
  for (int ii = 0; ii < 2; ++ii)
    for (int l = 0; l < 3; ++l) {
      double acc = 0;
      for (int jj = 0; jj < 2; ++jj)
        for (int m = 0; m < 3; ++m) acc += 2.0 * G2[ii][jj] * p.Tm[jj][m] * p.Sig[m][l];
      dTm[ii][l] = acc;
    }
  // Tm = J R
  double dJ[2][3];
  for (int ii = 0; ii < 2; ++ii)
    for (int l = 0; l < 3; ++l) {
      double acc = 0;
      for (int m = 0; m < 3; ++m) acc += dTm[ii][m] * k.R[l][m];
      dJ[ii][l] = acc;
    }
  // J00 = fx/z, J02 = -fx xr / z with xr = clamp(x/z); likewise row 1
  dpc[2] += dJ[0][0] * (-k.fx / (z * z)) + dJ[1][1] * (-k.fy / (z * z));
  if (p.clx) {
    dpc[2] += dJ[0][2] * (k.fx * p.xr / (z * z));
  } else {  // J02 = -fx x / z^2
    dpc[0] += dJ[0][2] * (-k.fx / (z * z));
    dpc[2] += dJ[0][2] * (2.0 * k.fx * x / (z * z * z));
  }
  if (p.cly) {
    dpc[2] += dJ[1][2] * (k.fy * p.yr / (z * z));
  } else {
    dpc[1] += dJ[1][2] * (-k.fy / (z * z));
    dpc[2] += dJ[1][2] * (2.0 * k.fy * y / (z * z * z));
  }
  // pc = R mu + t
  for (int j = 0; j < 3; ++j)
    for (int l = 0; l < 3; ++l) dmu[j] += k.R[l][j] * dpc[l];
  // Sig = M M^T with M = Rq diag(s)
  double M[3][3], dM[3][3];
  for (int l = 0; l < 3; ++l)
    for (int m = 0; m < 3; ++m) M[l][m] = p.Rq[l][m] * p.s[m];
  for (int l = 0; l < 3; ++l)
    for (int m = 0; m < 3; ++m) {
      double acc = 0;
      for (int n2 = 0; n2 < 3; ++n2) acc += (dSig[l][n2] + dSig[n2][l]) * M[n2][m];
      dM[l][m] = acc;
    }
  double dls[3], dRq[3][3];
  for (int m = 0; m < 3; ++m) {
    double acc = 0;
    for (int l = 0; l < 3; ++l) acc += dM[l][m] * p.Rq[l][m];
    dls[m] = acc * p.s[m];  // ds/dls = s
  }
  for (int l = 0; l < 3; ++l)
    for (int m = 0; m < 3; ++m) dRq[l][m] = dM[l][m] * p.s[m];
  // Rq(w, x, y, z) of the normalised quaternion
  const double w = p.qn[0], qx = p.qn[1], qy = p.qn[2], qz = p.qn[3];
  double dq[4];
  dq[0] = 2 * (-qz * dRq[0][1] + qy * dRq[0][2] + qz * dRq[1][0] - qx * dRq[1][2] - qy * dRq[2][0] +
               qx * dRq[2][1]);
  dq[1] = 2 * (qy * dRq[0][1] + qz * dRq[0][2] + qy * dRq[1][0] - 2 * qx * dRq[1][1] - w * dRq[1][2] +
               qz * dRq[2][0] + w * dRq[2][1] - 2 * qx * dRq[2][2]);
  dq[2] = 2 * (-2 * qy * dRq[0][0] + qx * dRq[0][1] + w * dRq[0][2] + qx * dRq[1][0] + qz * dRq[1][2] -
               w * dRq[2][0] + qz * dRq[2][1] - 2 * qy * dRq[2][2]);
  dq[3] = 2 * (-2 * qz * dRq[0][0] - w * dRq[0][1] + qx * dRq[0][2] + w * dRq[1][0] - 2 * qz * dRq[1][1] +
               qy * dRq[1][2] + qx * dRq[2][0] + qy * dRq[2][1]);
  // through q / |q|
  double dot = 0;
  for (int l = 0; l < 4; ++l) dot += p.qn[l] * dq[l];
  double dqraw[4];
  for (int l = 0; l < 4; ++l) dqraw[l] = (dq[l] - p.qn[l] * dot) / p.qlen;
  // colour: raw_c = sum_k sh[k][c] Y_k(d) + 0.5, clamped at 0
  double dd[3] = {0, 0, 0};
  for (int ch = 0; ch < 3; ++ch) {
    if (p.raw[ch] < 0) continue;
    const double gch = drgb[ch];
    for (int kk = 0; kk < 16; ++kk) {
      const int f = 3 * kk + ch;
      G(3 + f / 4, f % 4) += gch * p.Y[kk];
      for (int l = 0; l < 3; ++l) dd[l] += gch * g.sh[kk][ch] * p.dY[kk][l];
    }
  }
  double ddot = dd[0] * p.d[0] + dd[1] * p.d[1] + dd[2] * p.d[2];
  for (int l = 0; l < 3; ++l) dmu[l] += (dd[l] - p.d[l] * ddot) / p.dlen;
  // opacity = sigmoid(logit)
  const double dlogit = dopac * p.o * (1.0 - p.o);
  for (int l = 0; l < 3; ++l) G(0, l) += dmu[l];
  G(0, 3) += dlogit;
  for (int l = 0; l < 3; ++l) G(1, l) += dls[l];
  for (int l = 0; l < 4; ++l) G(2, l) += dqraw[l];
}

// ---------------------------------------------------------------- binning
// Each visible Gaussian is duplicated once per tile of its rectangle with key
// (tile id << 32) | float bits of depth, value = Gaussian index; the stable sort
// orders by (tile, depth, index).  Ranges [start, end) per tile, [0, 0) if empty.
int64_t bin_sort(const double* uvzo, const int32_t* radius, int64_t N, const Cam& k, uint64_t* keys,
                 uint32_t* vals, int64_t cap, uint32_t* ranges) {
  std::vector<std::pair<uint64_t, uint32_t>> inst;
  for (int64_t i = 0; i < N; ++i) {
    if (radius[i] <= 0) continue;
    int rect[4];
    rect_of(uvzo[4 * i + 0], uvzo[4 * i + 1], radius[i], k, rect);
    float zf = f32(uvzo[4 * i + 2]);
    uint32_t zb;
    std::memcpy(&zb, &zf, 4);
    for (int ty = rect[1]; ty < rect[3]; ++ty)
      for (int tx = rect[0]; tx < rect[2]; ++tx) {
        uint64_t tile = (uint64_t)ty * k.Tx + tx;
        inst.push_back({(tile << 32) | zb, (uint32_t)i});
      }
  }
  std::stable_sort(inst.begin(), inst.end(),
                   [](const std::pair<uint64_t, uint32_t>& l, const std::pair<uint64_t, uint32_t>& r) {
                     return l.first < r.first;
                   });
  const int64_t M = (int64_t)inst.size();
  const int64_t T = (int64_t)k.Tx * k.Ty;
  for (int64_t t = 0; t < 2 * T; ++t) ranges[t] = 0;
  if (M > cap) return M;
  for (int64_t j = 0; j < M; ++j) {
    if (keys) keys[j] = inst[j].first;
    vals[j] = inst[j].second;
    const uint64_t t = inst[j].first >> 32;
    if (j == 0 || (inst[j - 1].first >> 32) != t) ranges[2 * t] = (uint32_t)j;
    if (j == M - 1 || (inst[j + 1].first >> 32) != t) ranges[2 * t + 1] = (uint32_t)(j + 1);
  }
  return M;
}

// ---------------------------------------------------------------- render backward
// Reverse mode of composite_pixel for every pixel, summed per Gaussian.
// g2d: N x 9 = (du, dv, dA, dB, dC, dopacity, dr, dg, db), accumulated with +=.
void render_bwd(const View2D& in, const uint32_t* vals, const uint32_t* ranges, const Cam& k,
                const double bg[3], const double* dimg, double* g2d) {
  const int64_t P = (int64_t)k.W * k.H;
  for (int ty = 0; ty < k.Ty; ++ty)
    for (int tx = 0; tx < k.Tx; ++tx) {
      const int64_t t = (int64_t)ty * k.Tx + tx;
      for (int py = ty * TILE; py < std::min(ty * TILE + TILE, k.H); ++py)
        for (int px = tx * TILE; px < std::min(tx * TILE + TILE, k.W); ++px) {
          PixelResult pr = composite_pixel(in, vals, ranges[2 * t], ranges[2 * t + 1], px, py, true);
          const int64_t pix = (int64_t)py * k.W + px;
          const double dC[3] = {dimg[pix], dimg[P + pix], dimg[2 * P + pix]};
          // suffix: colour composited behind Gaussian j, plus the background
          double after[3] = {pr.T * bg[0], pr.T * bg[1], pr.T * bg[2]};
          for (int64_t n = (int64_t)pr.used.size() - 1; n >= 0; --n) {
            const Contrib& u = pr.used[n];
            const int64_t g = u.g;
            const double* col = in.rgb + 3 * g;
            double dalpha = 0;
            for (int c = 0; c < 3; ++c) {
              g2d[9 * g + 6 + c] += u.alpha * u.T * dC[c];
              dalpha += (u.T * col[c] - after[c] / (1.0 - u.alpha)) * dC[c];
            }
            for (int c = 0; c < 3; ++c) after[c] += u.alpha * u.T * col[c];
            if (u.clamped) continue;  // alpha = 0.99 does not depend on o or power
            const double o = in.uvzo[4 * g + 3];
            g2d[9 * g + 5] += dalpha * u.G;
            const double dpow = dalpha * o * u.G;
            const double A = in.conic[3 * g + 0], B = in.conic[3 * g + 1], Cc = in.conic[3 * g + 2];
            g2d[9 * g + 2] += dpow * (-0.5 * u.dx * u.dx);
            g2d[9 * g + 3] += dpow * (-u.dx * u.dy);
            g2d[9 * g + 4] += dpow * (-0.5 * u.dy * u.dy);
            // dx = px + 0.5 - u  =>  d power / du = A dx + B dy
            g2d[9 * g + 0] += dpow * (A * u.dx + B * u.dy);
            g2d[9 * g + 1] += dpow * (B * u.dx + Cc * u.dy);
          }
        }
    }
}

void render_fwd(const View2D& in, const uint32_t* vals, const uint32_t* ranges, const Cam& k,
                const double bg[3], double* img, double* T_final, uint32_t* n_contrib, double* margin) {
  const int64_t P = (int64_t)k.W * k.H;
  for (int ty = 0; ty < k.Ty; ++ty)
    for (int tx = 0; tx < k.Tx; ++tx) {
      const int64_t t = (int64_t)ty * k.Tx + tx;
      for (int py = ty * TILE; py < std::min(ty * TILE + TILE, k.H); ++py)
        for (int px = tx * TILE; px < std::min(tx * TILE + TILE, k.W); ++px) {
          PixelResult pr = composite_pixel(in, vals, ranges[2 * t], ranges[2 * t + 1], px, py, false);
          const int64_t pix = (int64_t)py * k.W + px;
          for (int c = 0; c < 3; ++c) img[c * P + pix] = pr.C[c] + pr.T * bg[c];
          if (T_final) T_final[pix] = pr.T;
          if (n_contrib) n_contrib[pix] = pr.n_contrib;
          if (margin) margin[pix] = pr.margin;
        }
    }
}

// ---------------------------------------------------------------- Adam
// Batch-scaled Adam (Grendel-GS notes §4.2): lr' = lr sqrt(b), beta' = beta^b,
// bias correction with beta'^t, eps after the square root.  Only the listed
// Gaussians change; their gradient is cleared afterwards.
void sparse_adam(double* p, double* gr, double* m, double* v, int64_t N, const uint32_t* idx, int64_t n_idx,
                 double lr, double beta1, double beta2, double eps, int batch, int64_t step) {
  const double b1 = std::pow(beta1, batch), b2 = std::pow(beta2, batch);
  const double lr_b = lr * std::sqrt((double)batch);
  const double bc1 = 1.0 - std::pow(b1, (double)step), bc2 = 1.0 - std::pow(b2, (double)step);
  for (int64_t n = 0; n < n_idx; ++n) {
    const int64_t i = idx[n];
    for (int plane = 0; plane < 15; ++plane)
      for (int lane = 0; lane < 4; ++lane) {
        const int64_t e = ((int64_t)plane * N + i) * 4 + lane;
        const double g = gr[e];
        m[e] = b1 * m[e] + (1.0 - b1) * g;
        v[e] = b2 * v[e] + (1.0 - b2) * g * g;
        const double mh = m[e] / bc1, vh = v[e] / bc2;
        p[e] -= lr_b * mh / (std::sqrt(vh) + eps);
        gr[e] = 0.0;
      }
  }
}

// ---------------------------------------------------------------- visible sets
// V_v = {i : radius_v[i] > 0}, ascending; U = union; inter = |V_i n V_j|;
// Jaccard = inter / |V_i u V_j| rounded to fp32 from the exact ratio, 0 for an
// empty union (Odin summary §1).
void visible_sets(const int32_t* radius, int B, int64_t N, int64_t* offsets, uint32_t* indices,
                  uint32_t* uni, int64_t* n_union, int64_t* inter, float* jac) {
  std::vector<std::vector<uint32_t>> sets(B);
  for (int b = 0; b < B; ++b)
    for (int64_t i = 0; i < N; ++i)
      if (radius[(int64_t)b * N + i] > 0) sets[b].push_back((uint32_t)i);
  offsets[0] = 0;
  for (int b = 0; b < B; ++b) {
    for (size_t n = 0; n < sets[b].size(); ++n) indices[offsets[b] + n] = sets[b][n];
    offsets[b + 1] = offsets[b] + (int64_t)sets[b].size();
  }
  int64_t nu = 0;
  for (int64_t i = 0; i < N; ++i) {
    bool any = false;
    for (int b = 0; b < B && !any; ++b) any = radius[(int64_t)b * N + i] > 0;
    if (any) uni[nu++] = (uint32_t)i;
  }
  *n_union = nu;
  for (int i = 0; i < B; ++i)
    for (int j = 0; j < B; ++j) {
      std::vector<uint32_t> out;
      std::set_intersection(sets[i].begin(), sets[i].end(), sets[j].begin(), sets[j].end(),
                            std::back_inserter(out));
      const int64_t n = (int64_t)out.size();
      const int64_t un = (int64_t)sets[i].size() + (int64_t)sets[j].size() - n;
      inter[i * B + j] = n;
      jac[i * B + j] = un == 0 ? 0.0f : (float)((double)n / (double)un);
    }
}

// Grendel-GS notes §3.1 (pixel-wise load balancing): the render time ET[i] of every 16x16
// pixel block, CumSum = cumsum(ET), a target of Total / K per GPU, split points by
// searchsorted.  The per-block "time" here is an integer cost (a per-pixel work count summed
// over the block), so the sums and the split points are exact.  Split k is the number of
// blocks whose inclusive cumulative cost is at most k Total / K (searchsorted on the right:
// a block that ends exactly on a target stays in the earlier part, so equal costs split
// equally), compared exactly as K C[i] <= k Total.  Part k holds tiles [bounds[k],
// bounds[k + 1]).
void tile_split(const uint32_t* cost_px, int W, int H, int K, uint64_t* tile_cost, uint64_t* cum, int64_t* bounds) {
  const int Tx = (W + 15) / 16, Ty = (H + 15) / 16;
  const int64_t T = (int64_t)Tx * Ty;
  for (int ty = 0; ty < Ty; ++ty)
    for (int tx = 0; tx < Tx; ++tx) {
      uint64_t s = 0;
      for (int y = ty * 16; y < std::min(H, ty * 16 + 16); ++y)
        for (int x = tx * 16; x < std::min(W, tx * 16 + 16); ++x) s += cost_px[(int64_t)y * W + x];
      tile_cost[(int64_t)ty * Tx + tx] = s;
    }
  uint64_t run = 0;
  for (int64_t i = 0; i < T; ++i) {
    run += tile_cost[i];
    cum[i] = run;
  }
  const uint64_t total = run;
  bounds[0] = 0;
  for (int k = 1; k < K; ++k) {
    int64_t c = 0;
    for (int64_t i = 0; i < T; ++i)
      if ((unsigned __int128)K * cum[i] <= (unsigned __int128)k * total) ++c;
    bounds[k] = c;
  }
  bounds[K] = T;
}

// Odin summary: the relative locality graph over views with Jaccard edge weights w_uv, and
// the scheduling score s(v | U_prev) = sum of w_uv over the previous set U_prev; static
// data scheduling orders the task units so that weakly coupled transitions follow one
// another.  Views are taken one at a time into task units of `unit` views; the next view is
// the unscheduled one with the smallest score against the previous unit (ties: the lower
// index), the first unit's scores being 0.  The scores are float32 sums over the previous
// unit in its scheduling order -- the precision and order the kernel decides in.
void view_order(const float* w, int B, int unit, int32_t* order, float* score) {
  std::vector<int> prev, cur;
  std::vector<char> done(B, 0);
  for (int k = 0; k < B; ++k) {
    int best = -1;
    float best_s = 0.f;
    for (int v = 0; v < B; ++v) {
      if (done[v]) continue;
      float s = 0.f;
      for (int u : prev) s += w[(int64_t)u * B + v];
      if (best < 0 || s < best_s) {
        best = v;
        best_s = s;
      }
    }
    done[best] = 1;
    order[k] = best;
    score[k] = best_s;
    cur.push_back(best);
    if ((int)cur.size() == unit) {
      prev = cur;
      cur.clear();
    }
  }
}

// Grendel-GS notes, 训练流程 (densification: "prune low-opacity Gaussians"): keep Gaussian i
// when its opacity logit (plane 0, w) is at least min_logit -- sigmoid is increasing, so
// this is opacity >= sigmoid(min_logit) -- and copy its 15 parameter planes and both Adam
// moment planes to the next free slot, in index order.  planes: `n_sets` arrays of
// [15][n][4]; out: the same sets as [15][out_stride][4].  Returns the number kept.
int64_t prune(const float* const* planes, int n_sets, int64_t n, float min_logit, float* const* out,
              int64_t out_stride) {
  int64_t k = 0;
  for (int64_t i = 0; i < n; ++i) {
    const float logit = planes[0][(0 * n + i) * 4 + 3];
    if (!(logit >= min_logit)) continue;
    if (k < out_stride)
      for (int s = 0; s < n_sets; ++s)
        for (int pl = 0; pl < 15; ++pl)
          for (int c = 0; c < 4; ++c) out[s][((int64_t)pl * out_stride + k) * 4 + c] = planes[s][((int64_t)pl * n + i) * 4 + c];
    ++k;
  }
  return k;
}

// Grendel-GS notes, 训练流程 ("致密化": clone or split the Gaussians that need more detail,
// prune the transparent ones).  The pages give no criterion; the readings taken:
//  * statistic: per Gaussian, the sum over the views that see it (radius > 0) of the length of
//    its screen-space mean gradient |(dL/du, dL/dv)| in that view, and the number of those
//    views (densify_stat);
//  * selected: seen at least once and sum / count >= grad_threshold, compared in fp32 (the
//    precision the kernel decides in);
//  * split if the largest log-scale exceeds log_scale_threshold (compared in fp32, no exp
//    evaluated), else clone;
//  * the output: the Gaussians not split, in index order, then for every selected Gaussian in
//    index order its new ones: a clone (an exact copy), or two split children with means
//    mu + R(q / |q|) (s * z_k) (s = exp(log-scale), z_k the caller's standard normals k = 0, 1)
//    and log-scales lowered by ln 1.6, the other parameters copied; new Gaussians start with
//    zero Adam moments, kept ones keep theirs.
void densify_stat(const double* g2d, const int32_t* radius, int64_t N, double* stat) {
  for (int64_t i = 0; i < N; ++i) {
    if (radius[i] <= 0) continue;
    const double du = g2d[9 * i + 0], dv = g2d[9 * i + 1];
    stat[2 * i + 0] += std::sqrt(du * du + dv * dv);
    stat[2 * i + 1] += 1.0;
  }
}

void quat_rotation(const double q[4], double R[3][3]) {
  const double len = std::sqrt(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]);
  const double w = q[0] / len, x = q[1] / len, y = q[2] / len, z = q[3] / len;
  R[0][0] = 1 - 2 * (y * y + z * z); R[0][1] = 2 * (x * y - w * z);     R[0][2] = 2 * (x * z + w * y);
  R[1][0] = 2 * (x * y + w * z);     R[1][1] = 1 - 2 * (x * x + z * z); R[1][2] = 2 * (y * z - w * x);
  R[2][0] = 2 * (x * z - w * y);     R[2][1] = 2 * (y * z + w * x);     R[2][2] = 1 - 2 * (x * x + y * y);
}

int64_t densify(const float* params, const float* m, const float* v, const float* stat, int64_t N,
                float grad_threshold, float log_scale_threshold, const float* normals, double* out_p,
                double* out_m, double* out_v, int64_t out_stride, int64_t* n_clone, int64_t* n_split) {
  auto at = [&](const float* a, int pl, int64_t i, int c) { return (double)a[((int64_t)pl * N + i) * 4 + c]; };
  std::vector<int> kind(N, 0);  // 0 untouched, 1 clone, 2 split
  int64_t clones = 0, splits = 0;
  for (int64_t i = 0; i < N; ++i) {
    const float sum = stat[2 * i], cnt = stat[2 * i + 1];
    if (!(cnt > 0.0f)) continue;
    const float avg = sum / cnt;
    if (!(avg >= grad_threshold)) continue;
    const float lmax = std::max(std::max(params[(1 * N + i) * 4 + 0], params[(1 * N + i) * 4 + 1]),
                                params[(1 * N + i) * 4 + 2]);
    kind[i] = lmax > log_scale_threshold ? 2 : 1;
    if (kind[i] == 2) ++splits; else ++clones;
  }
  *n_clone = clones;
  *n_split = splits;
  const int64_t n_out = N - splits + clones + 2 * splits;
  int64_t k = 0;
  auto put = [&](int64_t dst, const double p[15][4], bool keep_moments, int64_t src) {
    if (dst >= out_stride) return;
    for (int pl = 0; pl < 15; ++pl)
      for (int c = 0; c < 4; ++c) {
        out_p[((int64_t)pl * out_stride + dst) * 4 + c] = p[pl][c];
        out_m[((int64_t)pl * out_stride + dst) * 4 + c] = keep_moments ? at(m, pl, src, c) : 0.0;
        out_v[((int64_t)pl * out_stride + dst) * 4 + c] = keep_moments ? at(v, pl, src, c) : 0.0;
      }
  };
  double p[15][4];
  for (int64_t i = 0; i < N; ++i) {  // the Gaussians not split, in index order
    if (kind[i] == 2) continue;
    for (int pl = 0; pl < 15; ++pl)
      for (int c = 0; c < 4; ++c) p[pl][c] = at(params, pl, i, c);
    put(k++, p, true, i);
  }
  for (int64_t i = 0; i < N; ++i) {  // then the new ones of every selected Gaussian
    if (kind[i] == 0) continue;
    for (int pl = 0; pl < 15; ++pl)
      for (int c = 0; c < 4; ++c) p[pl][c] = at(params, pl, i, c);
    if (kind[i] == 1) {
      put(k++, p, false, i);
      continue;
    }
    double q[4] = {p[2][0], p[2][1], p[2][2], p[2][3]}, R[3][3];
    quat_rotation(q, R);
    const double s[3] = {std::exp(p[1][0]), std::exp(p[1][1]), std::exp(p[1][2])};
    for (int child = 0; child < 2; ++child) {
      double c[15][4];
      std::memcpy(c, p, sizeof(c));
      for (int r = 0; r < 3; ++r) {
        double off = 0;
        for (int j = 0; j < 3; ++j) off += R[r][j] * s[j] * (double)normals[6 * i + 3 * child + j];
        c[0][r] = p[0][r] + off;
      }
      for (int j = 0; j < 3; ++j) c[1][j] = p[1][j] - std::log(1.6);
      put(k++, c, false, i);
    }
  }
  return n_out;
}

}  // namespace

// ======================================================================= C ABI
extern "C" {

// Projection of N Gaussians.  params: [15][N][4] doubles.  cam: 17 doubles
// (R row-major, t, fx, fy, cx, cy, znear).  Outputs (any may be null except
// uvzo / conic / radius / rgb): uvzo N x 4, conic N x 3, radius N, rgb N x 3,
// rect N x 4, tiles N, raw N x 3 (colour before the clamp), margin N (relative margin of the
// nearest decision that can change an output: culls, and the tile rectangle -- through the
// screen position or the radius -- where it adds or drops a tile the Gaussian reaches),
// rmargin N (relative margin of the radius ceiling; 0 where a floor of the screen position
// within its rounding bound would give another rectangle: the values that may differ).
void oracle_project(const double* params, int64_t N, const double* cam, int W, int H, double* uvzo,
                    double* conic, int32_t* radius, double* rgb, int32_t* rect, int32_t* tiles, double* raw,
                    double* margin, double* rmargin) {
  const Cam k = load_cam(cam, W, H);
  for (int64_t i = 0; i < N; ++i) {
    const Proj p = project_one(load_gauss(params, N, i), k);
    const bool v = p.vis;
    uvzo[4 * i + 0] = v ? p.u : 0; uvzo[4 * i + 1] = v ? p.v : 0;
    uvzo[4 * i + 2] = v ? p.z : 0; uvzo[4 * i + 3] = v ? p.o : 0;
    for (int l = 0; l < 3; ++l) conic[3 * i + l] = v ? p.conic[l] : 0;
    radius[i] = v ? p.r : 0;
    for (int l = 0; l < 3; ++l) rgb[3 * i + l] = v ? p.rgb[l] : 0;
    if (rect)
      for (int l = 0; l < 4; ++l) rect[4 * i + l] = v ? p.rect[l] : 0;
    if (tiles) tiles[i] = v ? p.tiles : 0;
    if (raw)
      for (int l = 0; l < 3; ++l) raw[3 * i + l] = v ? p.raw[l] : 0;
    if (margin) margin[i] = p.margin;
    if (rmargin) rmargin[i] = v ? p.rmargin : 1e30;
  }
}

// Binning: returns M (instances).  keys may be null.  ranges: T x 2.
int64_t oracle_bin_sort(const double* uvzo, const int32_t* radius, int64_t N, int W, int H, uint64_t* keys,
                        uint32_t* vals, int64_t cap, uint32_t* ranges) {
  double dummy[17] = {0};
  Cam k = load_cam(dummy, W, H);
  return bin_sort(uvzo, radius, N, k, keys, vals, cap, ranges);
}

void oracle_render_fwd(const double* uvzo, const double* conic, const double* rgb, const uint32_t* vals,
                       const uint32_t* ranges, int W, int H, const double* bg, double* img, double* T_final,
                       uint32_t* n_contrib, double* margin) {
  double dummy[17] = {0};
  Cam k = load_cam(dummy, W, H);
  View2D in{uvzo, conic, rgb};
  render_fwd(in, vals, ranges, k, bg, img, T_final, n_contrib, margin);
}

// Per-pixel work of the compositing walk, [H][W] each: n_eval = list entries evaluated (through
// the one whose transmittance would fall below 1e-4, else the whole tile list), n_used = entries
// accumulated.
void oracle_render_counts(const double* uvzo, const double* conic, const double* rgb, const uint32_t* vals,
                          const uint32_t* ranges, int W, int H, uint32_t* n_eval, uint32_t* n_used) {
  double dummy[17] = {0};
  Cam k = load_cam(dummy, W, H);
  View2D in{uvzo, conic, rgb};
  for (int py = 0; py < H; ++py)
    for (int px = 0; px < W; ++px) {
      const int64_t t = (int64_t)(py / TILE) * k.Tx + px / TILE;
      const PixelResult pr = composite_pixel(in, vals, ranges[2 * t], ranges[2 * t + 1], px, py, false);
      n_eval[(int64_t)py * W + px] = pr.n_eval;
      n_used[(int64_t)py * W + px] = pr.n_used;
    }
}

// g2d: N x 9, accumulated (+=).
void oracle_render_bwd(const double* uvzo, const double* conic, const double* rgb, const uint32_t* vals,
                       const uint32_t* ranges, int W, int H, const double* bg, const double* dimg, double* g2d) {
  double dummy[17] = {0};
  Cam k = load_cam(dummy, W, H);
  View2D in{uvzo, conic, rgb};
  render_bwd(in, vals, ranges, k, bg, dimg, g2d);
}

// Returns scale * (w_l1 L1 + w_ssim (1 - SSIM)); dimg (3 x H x W) may be null.
double oracle_loss(const double* img, const double* tgt, int W, int H, double w_l1, double w_ssim, double scale,
                   double* dimg) {
  return loss_one(img, tgt, W, H, w_l1, w_ssim, scale, dimg);
}

// Projection backward: g2d N x 9 as produced by oracle_render_bwd; grads [15][N][4] (+=).
void oracle_project_bwd(const double* params, int64_t N, const double* cam, int W, int H, const double* g2d,
                        double* grads) {
  const Cam k = load_cam(cam, W, H);
  for (int64_t i = 0; i < N; ++i) {
    const Gauss g = load_gauss(params, N, i);
    const Proj p = project_one(g, k);
    const double* q = g2d + 9 * i;
    project_bwd_one(g, p, k, q[0], q[1], q + 2, q[5], q + 6, grads, N, i);
  }
}

void oracle_sparse_adam(double* params, double* grads, double* m, double* v, int64_t N, const uint32_t* idx,
                        int64_t n_idx, double lr, double beta1, double beta2, double eps, int batch,
                        int64_t step) {
  sparse_adam(params, grads, m, v, N, idx, n_idx, lr, beta1, beta2, eps, batch, step);
}

void oracle_visible_sets(const int32_t* radius, int B, int64_t N, int64_t* offsets, uint32_t* indices,
                         uint32_t* uni, int64_t* n_union, int64_t* inter, float* jac) {
  visible_sets(radius, B, N, offsets, indices, uni, n_union, inter, jac);
}

// Per-tile costs, their inclusive cumulative sum and the K + 1 split points (Grendel-GS
// notes §3.1).  cost_px: H x W.  tile_cost, cum: ceil(W/16) ceil(H/16).  bounds: K + 1.
void oracle_tile_split(const uint32_t* cost_px, int W, int H, int K, uint64_t* tile_cost, uint64_t* cum,
                       int64_t* bounds) {
  tile_split(cost_px, W, H, K, tile_cost, cum, bounds);
}

// Greedy view order by the Odin scheduling score.  w: B x B float32 weights (Jaccard).
void oracle_view_order(const float* w, int B, int unit, int32_t* order, float* score) {
  view_order(w, B, unit, order, score);
}

// Densification statistic of one view (+= into stat, N x 2: sum of |(du, dv)|, views).
void oracle_densify_stat(const double* g2d, const int32_t* radius, int64_t N, double* stat) {
  densify_stat(g2d, radius, N, stat);
}

// Clone / split (readings above densify_stat).  params, m, v: float32 [15][N][4]; stat:
// float32 N x 2; normals: float32 N x 6.  Outputs [15][out_stride][4] doubles (slots past
// out_stride not written).  Returns the output count; n_clone / n_split receive the counts.
int64_t oracle_densify(const float* params, const float* m, const float* v, const float* stat, int64_t N,
                       float grad_threshold, float log_scale_threshold, const float* normals, double* out_p,
                       double* out_m, double* out_v, int64_t out_stride, int64_t* n_clone, int64_t* n_split) {
  return densify(params, m, v, stat, N, grad_threshold, log_scale_threshold, normals, out_p, out_m, out_v,
                 out_stride, n_clone, n_split);
}

// Opacity pruning: planes / out are arrays of n_sets pointers (parameters, then moments).
int64_t oracle_prune(const float* const* planes, int n_sets, int64_t n, float min_logit, float* const* out,
                     int64_t out_stride) {
  return prune(planes, n_sets, n, min_logit, out, out_stride);
}

// One whole training step over B views.  cams: B x 17.  targets: B x 3 x H x W.
// grads_out ([15][N][4], may be null) receives the batch gradient before the
// update; params / m / v are updated in place when do_adam != 0.
// Returns the batch loss (mean of the per-view losses).
double oracle_step(double* params, double* m, double* v, int64_t N, const double* cams, int B, int W, int H,
                   const double* targets, const double* bg, double w_l1, double w_ssim, double lr, double beta1,
                   double beta2, double eps, int64_t step, int do_adam, double* grads_out, double* images_out) {
  const int64_t P = (int64_t)W * H;
  const int64_t NF = 15 * N * 4;
  std::vector<double> grads(NF, 0.0);
  std::vector<int32_t> radii((size_t)B * N);
  double loss = 0;
  for (int b = 0; b < B; ++b) {
    const Cam k = load_cam(cams + 17 * b, W, H);
    std::vector<double> uvzo(4 * N), conic(3 * N), rgb(3 * N);
    std::vector<Gauss> gs(N);
    std::vector<Proj> ps(N);
    for (int64_t i = 0; i < N; ++i) {
      gs[i] = load_gauss(params, N, i);
      ps[i] = project_one(gs[i], k);
      const Proj& p = ps[i];
      uvzo[4 * i + 0] = p.u; uvzo[4 * i + 1] = p.v; uvzo[4 * i + 2] = p.z; uvzo[4 * i + 3] = p.vis ? p.o : 0;
      for (int l = 0; l < 3; ++l) { conic[3 * i + l] = p.vis ? p.conic[l] : 0; rgb[3 * i + l] = p.rgb[l]; }
      radii[(size_t)b * N + i] = p.vis ? p.r : 0;
    }
    int64_t cap = 0;
    for (int64_t i = 0; i < N; ++i) cap += ps[i].vis ? ps[i].tiles : 0;
    std::vector<uint32_t> vals(std::max<int64_t>(cap, 1)), ranges(2 * (int64_t)k.Tx * k.Ty);
    bin_sort(uvzo.data(), radii.data() + (size_t)b * N, N, k, nullptr, vals.data(), cap, ranges.data());
    View2D in{uvzo.data(), conic.data(), rgb.data()};
    std::vector<double> img(3 * P), dimg(3 * P), g2d(9 * N, 0.0);
    render_fwd(in, vals.data(), ranges.data(), k, bg, img.data(), nullptr, nullptr, nullptr);
    if (images_out) std::copy(img.begin(), img.end(), images_out + (int64_t)b * 3 * P);
    loss += loss_one(img.data(), targets + (int64_t)b * 3 * P, W, H, w_l1, w_ssim, 1.0 / B, dimg.data());
    render_bwd(in, vals.data(), ranges.data(), k, bg, dimg.data(), g2d.data());
    for (int64_t i = 0; i < N; ++i) {
      const double* q = g2d.data() + 9 * i;
      project_bwd_one(gs[i], ps[i], k, q[0], q[1], q + 2, q[5], q + 6, grads.data(), N, i);
    }
  }
  if (grads_out) std::copy(grads.begin(), grads.end(), grads_out);
  if (do_adam) {
    std::vector<uint32_t> uni;
    for (int64_t i = 0; i < N; ++i) {
      bool any = false;
      for (int b = 0; b < B && !any; ++b) any = radii[(size_t)b * N + i] > 0;
      if (any) uni.push_back((uint32_t)i);
    }
    sparse_adam(params, grads.data(), m, v, N, uni.data(), (int64_t)uni.size(), lr, beta1, beta2, eps, B, step);
  }
  return loss;
}

// Real SH basis and its gradient at unit direction d (for the basis pins).
void oracle_sh_basis(const double* d, double* Y, double* dY) {
  double dYl[16][3];
  sh_basis(d, Y, dYl);
  for (int k = 0; k < 16; ++k)
    for (int l = 0; l < 3; ++l) dY[3 * k + l] = dYl[k][l];
}

}  // extern "C"
