// Projection of 3D Gaussians to screen space and its reverse mode (gs_project, gs_project_bwd).
//
// "Transform" step of the Grendel-GS training flow (训练流程): each Gaussian -> 2D position,
// depth, footprint radius and view-dependent colour.  One thread per Gaussian; every
// parameter plane is read as one coalesced float4 per thread (512 B per warp), the SH
// planes only for Gaussians that survive the culls.  HBM-bound: 240 B read + 48 B written
// per visible Gaussian, 16 B read per culled one.
#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace {

using gs::Cam;

// Real SH basis, degree <= 3, k = l*l + l + m (real part of Y_l^m with the
// Condon-Shortley phase, times sqrt2 for m != 0; Im for m < 0).
constexpr float kC0 = 0.28209479177387814f;
constexpr float kC1 = 0.4886025119029199f;
constexpr float kA2 = 1.0925484305920792f;   // sqrt(15/pi)/2
constexpr float kB2 = 0.31539156525252005f;  // sqrt(5/pi)/4
constexpr float kC2 = 0.5462742152960396f;   // sqrt(15/pi)/4
constexpr float kE3 = 0.5900435899266435f;   // sqrt(35/(2pi))/4
constexpr float kF3 = 2.890611442640554f;    // sqrt(105/pi)/2
constexpr float kG3 = 0.4570457994644658f;   // sqrt(21/(2pi))/4
constexpr float kH3 = 0.3731763325901154f;   // sqrt(7/pi)/4
constexpr float kI3 = 1.445305721320277f;    // sqrt(105/pi)/4

struct SHBasis {
  float y[16];
};

__device__ __forceinline__ void sh_eval(float x, float y, float z, SHBasis& b) {
  const float xx = x * x, yy = y * y, zz = z * z;
  b.y[0] = kC0;
  b.y[1] = -kC1 * y;
  b.y[2] = kC1 * z;
  b.y[3] = -kC1 * x;
  b.y[4] = kA2 * x * y;
  b.y[5] = -kA2 * y * z;
  b.y[6] = kB2 * (2.f * zz - xx - yy);
  b.y[7] = -kA2 * x * z;
  b.y[8] = kC2 * (xx - yy);
  b.y[9] = -kE3 * y * (3.f * xx - yy);
  b.y[10] = kF3 * x * y * z;
  b.y[11] = -kG3 * y * (4.f * zz - xx - yy);
  b.y[12] = kH3 * z * (2.f * zz - 3.f * xx - 3.f * yy);
  b.y[13] = -kG3 * x * (4.f * zz - xx - yy);
  b.y[14] = kI3 * z * (xx - yy);
  b.y[15] = -kE3 * x * (xx - 3.f * yy);
}

// Gradient of sum_k w[k] Y_k with respect to the (unnormalised) direction components.
__device__ __forceinline__ float3 sh_grad_dot(float x, float y, float z, const float* w) {
  const float xx = x * x, yy = y * y, zz = z * z;
  float gx = 0.f, gy = 0.f, gz = 0.f;
  // l = 1
  gy += -kC1 * w[1];
  gz += kC1 * w[2];
  gx += -kC1 * w[3];
  // l = 2
  gx += kA2 * y * w[4];            gy += kA2 * x * w[4];
  gy += -kA2 * z * w[5];           gz += -kA2 * y * w[5];
  gx += -2.f * kB2 * x * w[6];     gy += -2.f * kB2 * y * w[6];    gz += 4.f * kB2 * z * w[6];
  gx += -kA2 * z * w[7];           gz += -kA2 * x * w[7];
  gx += 2.f * kC2 * x * w[8];      gy += -2.f * kC2 * y * w[8];
  // l = 3
  gx += -6.f * kE3 * x * y * w[9];  gy += -3.f * kE3 * (xx - yy) * w[9];
  gx += kF3 * y * z * w[10];        gy += kF3 * x * z * w[10];       gz += kF3 * x * y * w[10];
  gx += 2.f * kG3 * x * y * w[11];  gy += -kG3 * (4.f * zz - xx - 3.f * yy) * w[11];  gz += -8.f * kG3 * y * z * w[11];
  gx += -6.f * kH3 * x * z * w[12]; gy += -6.f * kH3 * y * z * w[12];  gz += kH3 * (6.f * zz - 3.f * xx - 3.f * yy) * w[12];
  gx += -kG3 * (4.f * zz - 3.f * xx - yy) * w[13];  gy += 2.f * kG3 * x * y * w[13];  gz += -8.f * kG3 * x * z * w[13];
  gx += 2.f * kI3 * x * z * w[14];  gy += -2.f * kI3 * y * z * w[14];  gz += kI3 * (xx - yy) * w[14];
  gx += -3.f * kE3 * (xx - yy) * w[15];  gy += 6.f * kE3 * x * y * w[15];
  return make_float3(gx, gy, gz);
}

// Everything the forward computes for one Gaussian, kept for the reverse pass.
struct Fwd {
  float px, py, pz;       // camera-space mean
  float s[3];             // scales
  float opac;
  float qn[4], qinv;      // normalised quaternion, 1/|q|
  float Rq[9];            // rotation of the normalised quaternion
  float Sg[6];            // Sigma: xx, xy, xz, yy, yz, zz
  float xr, yr;           // clamped x/z, y/z
  bool clx, cly;
  float T0[3], T1[3];     // rows of J W
  float a, b, c, det;     // dilated 2D covariance and its determinant
  float A, B, C;          // conic
  float u, v;
  int radius, x0, y0, x1, y1;
};

// Where a Gaussian's parameter planes are read from: global memory (plane pl of Gaussian i
// at params[pl][i]) or a shared-memory copy ([pl][thread]).
struct GlobalParams {
  const float* p;
  int64_t n, i;
  __device__ __forceinline__ float4 plane(int pl) const { return ldg4(p, (int64_t)pl * n + i); }
};
template <int kThreadsPerCta>
struct SharedParams {
  const float4* s;
  int t;
  __device__ __forceinline__ float4 plane(int pl) const { return s[pl * kThreadsPerCta + t]; }
};

// The view-independent part of the forward: scales, opacity, normalised quaternion, its
// rotation and the 3-D covariance.
template <class Src>
__device__ __forceinline__ void project_intrinsics(const Src& src, Fwd& f) {
  const float4 p0 = src.plane(0);
  const float4 p1 = src.plane(1);
  const float4 p2 = src.plane(2);
  f.s[0] = expf(p1.x);
  f.s[1] = expf(p1.y);
  f.s[2] = expf(p1.z);
  f.opac = 1.f / (1.f + expf(-p0.w));
  const float qq = p2.x * p2.x + p2.y * p2.y + p2.z * p2.z + p2.w * p2.w;
  f.qinv = rsqrtf(qq);
  const float w = p2.x * f.qinv, x = p2.y * f.qinv, y = p2.z * f.qinv, z = p2.w * f.qinv;
  f.qn[0] = w; f.qn[1] = x; f.qn[2] = y; f.qn[3] = z;
  f.Rq[0] = 1.f - 2.f * (y * y + z * z); f.Rq[1] = 2.f * (x * y - w * z);       f.Rq[2] = 2.f * (x * z + w * y);
  f.Rq[3] = 2.f * (x * y + w * z);       f.Rq[4] = 1.f - 2.f * (x * x + z * z); f.Rq[5] = 2.f * (y * z - w * x);
  f.Rq[6] = 2.f * (x * z - w * y);       f.Rq[7] = 2.f * (y * z + w * x);       f.Rq[8] = 1.f - 2.f * (x * x + y * y);
  float M[9];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int c = 0; c < 3; ++c) M[3 * r + c] = f.Rq[3 * r + c] * f.s[c];
  f.Sg[0] = M[0] * M[0] + M[1] * M[1] + M[2] * M[2];
  f.Sg[1] = M[0] * M[3] + M[1] * M[4] + M[2] * M[5];
  f.Sg[2] = M[0] * M[6] + M[1] * M[7] + M[2] * M[8];
  f.Sg[3] = M[3] * M[3] + M[4] * M[4] + M[5] * M[5];
  f.Sg[4] = M[3] * M[6] + M[4] * M[7] + M[5] * M[8];
  f.Sg[5] = M[6] * M[6] + M[7] * M[7] + M[8] * M[8];
}

// The view-dependent part, on a Fwd whose intrinsics are set.  Returns false if the Gaussian
// is culled in this view.
template <class Src>
__device__ __forceinline__ bool project_view(const Src& src, const Cam& k, Fwd& f) {
  const float4 p0 = src.plane(0);
  f.px = k.R[0] * p0.x + k.R[1] * p0.y + k.R[2] * p0.z + k.t[0];
  f.py = k.R[3] * p0.x + k.R[4] * p0.y + k.R[5] * p0.z + k.t[1];
  f.pz = k.R[6] * p0.x + k.R[7] * p0.y + k.R[8] * p0.z + k.t[2];
  if (!(f.pz > k.znear)) return false;
  const float iz = 1.f / f.pz;
  const float limx = 1.3f * (0.5f * (float)k.W / k.fx), limy = 1.3f * (0.5f * (float)k.H / k.fy);
  const float rx = f.px * iz, ry = f.py * iz;
  f.clx = rx < -limx || rx > limx;
  f.cly = ry < -limy || ry > limy;
  f.xr = fminf(fmaxf(rx, -limx), limx);
  f.yr = fminf(fmaxf(ry, -limy), limy);
  const float jx = k.fx * iz, jy = k.fy * iz;
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    f.T0[c] = jx * (k.R[c] - f.xr * k.R[6 + c]);
    f.T1[c] = jy * (k.R[3 + c] - f.yr * k.R[6 + c]);
  }
  // (J W) Sigma (J W)^T
  const float* S = f.Sg;
  const float s0x = S[0] * f.T0[0] + S[1] * f.T0[1] + S[2] * f.T0[2];
  const float s0y = S[1] * f.T0[0] + S[3] * f.T0[1] + S[4] * f.T0[2];
  const float s0z = S[2] * f.T0[0] + S[4] * f.T0[1] + S[5] * f.T0[2];
  const float s1x = S[0] * f.T1[0] + S[1] * f.T1[1] + S[2] * f.T1[2];
  const float s1y = S[1] * f.T1[0] + S[3] * f.T1[1] + S[4] * f.T1[2];
  const float s1z = S[2] * f.T1[0] + S[4] * f.T1[1] + S[5] * f.T1[2];
  f.a = f.T0[0] * s0x + f.T0[1] * s0y + f.T0[2] * s0z + 0.3f;
  f.b = f.T0[0] * s1x + f.T0[1] * s1y + f.T0[2] * s1z;
  f.c = f.T1[0] * s1x + f.T1[1] * s1y + f.T1[2] * s1z + 0.3f;
  f.det = f.a * f.c - f.b * f.b;
  if (!(f.det > 0.f)) return false;
  const float idet = 1.f / f.det;
  f.A = f.c * idet;
  f.B = -f.b * idet;
  f.C = f.a * idet;
  const float mid = 0.5f * (f.a + f.c);
  const float lam = mid + sqrtf(fmaxf(mid * mid - f.det, 0.f));
  const float rr = ceilf(3.f * sqrtf(lam));
  f.radius = rr < 16777216.f ? (int)rr : 16777216;  // radii beyond 2^24 px cover every tile anyway
  f.u = k.fx * f.px * iz + k.cx;
  f.v = k.fy * f.py * iz + k.cy;
  // tile rectangle: floor((u -+ r)/16) in integer form (exact for any float u)
  const int fu = (int)floorf(fminf(fmaxf(f.u, -1e9f), 1e9f));
  const int fv = (int)floorf(fminf(fmaxf(f.v, -1e9f), 1e9f));
  const int r = f.radius;
  f.x0 = min(max((fu - r) >> 4, 0), k.Tx);
  f.x1 = min(max(((fu + r) >> 4) + 1, 0), k.Tx);
  f.y0 = min(max((fv - r) >> 4, 0), k.Ty);
  f.y1 = min(max(((fv + r) >> 4) + 1, 0), k.Ty);
  return f.x0 < f.x1 && f.y0 < f.y1;
}

// The whole forward of one Gaussian in one view.  Returns false if it is culled.
template <class Src>
__device__ __forceinline__ bool project_core(const Src& src, const Cam& k, Fwd& f) {
  const float4 p0 = src.plane(0);
  const float pz = k.R[6] * p0.x + k.R[7] * p0.y + k.R[8] * p0.z + k.t[2];
  if (!(pz > k.znear)) return false;  // the near-plane cull needs only the mean
  project_intrinsics(src, f);
  return project_view(src, k, f);
}

// Colour and the three records of Gaussian i in a view that does not cull it.
template <class Src>
__device__ __forceinline__ void emit_projection(const Src& src, const Fwd& f, float3 campos, float* __restrict__ proj,
                                                int64_t n, int64_t i) {
  {
    const float4 p0 = src.plane(0);
    float dx = p0.x - campos.x, dy = p0.y - campos.y, dz = p0.z - campos.z;
    const float il = rsqrtf(dx * dx + dy * dy + dz * dz);
    dx *= il; dy *= il; dz *= il;
    SHBasis b;
    sh_eval(dx, dy, dz, b);
    float rgb[3] = {0.5f, 0.5f, 0.5f};
#pragma unroll
    for (int pl = 0; pl < 12; ++pl) {
      const float4 s = src.plane(3 + pl);
      const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int l = 0; l < 4; ++l) {
        const int fidx = 4 * pl + l;  // 3 * coefficient + channel
        rgb[fidx % 3] += sv[l] * b.y[fidx / 3];
      }
    }
    st4(proj, i, make_float4(f.u, f.v, f.pz, f.opac));
    st4(proj, n + i, make_float4(f.A, f.B, f.C, __int_as_float(f.radius)));
    st4(proj, 2 * n + i, make_float4(fmaxf(rgb[0], 0.f), fmaxf(rgb[1], 0.f), fmaxf(rgb[2], 0.f),
                                     __int_as_float((f.x1 - f.x0) * (f.y1 - f.y0))));
  }
}

// Zero records: Gaussian i is culled in this view.
__device__ __forceinline__ void emit_culled(float* __restrict__ proj, int64_t n, int64_t i) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  st4(proj, i, z);
  st4(proj, n + i, z);
  st4(proj, 2 * n + i, z);
}

__global__ void __launch_bounds__(256) k_project_fwd(const float* __restrict__ params, int64_t n, Cam k,
                                                     float3 campos, float* __restrict__ proj) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  Fwd f;
  const GlobalParams src{params, n, i};
  if (project_core(src, k, f)) emit_projection(src, f, campos, proj, n, i);
  else emit_culled(proj, n, i);
}

// Up to 16 views of one batch in one launch: the parameters are read once and the
// view-independent part (scales, opacity, rotation, 3-D covariance) is computed once, at the
// first view that does not cull the Gaussian at the near plane.
constexpr int kMaxProjViews = 16;
struct ProjViews {
  Cam k[kMaxProjViews];
  float3 campos[kMaxProjViews];
  float* proj[kMaxProjViews];
  uint32_t* bits;        // optional visibility bitsets of the launch's views, [batch][bits_stride]
  int64_t bits_stride;
  int64_t bits_words;    // ceil(n / 32)
  int batch;
};

// The batch kernel's parameter source: planes 0-2 from global memory, the twelve SH planes
// from the thread's shared-memory copy ([plane][thread]; every visible view reads them).
constexpr int kProjThreads = 256;
struct StagedSH {
  const float* p;
  int64_t n, i;
  const float4* sh;
  int t;
  __device__ __forceinline__ float4 plane(int pl) const {
    return pl < 3 ? ldg4(p, (int64_t)pl * n + i) : sh[(pl - 3) * kProjThreads + t];
  }
};

__global__ void __launch_bounds__(kProjThreads, 4) k_project_fwd_batch(const float* __restrict__ params, int64_t n,
                                                                    const __grid_constant__ ProjViews pv) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float4* sh = reinterpret_cast<float4*>(smem_raw);  // [12][kProjThreads], thread-private slots
  const int t = threadIdx.x;
  const int64_t i = (int64_t)blockIdx.x * kProjThreads + t;
  const bool live = i < n;
  if (!live && !pv.bits) return;  // (with bitsets every lane of a warp takes part in the ballot)
  const GlobalParams src{params, n, i};
  const StagedSH staged{params, n, i, sh, t};
  const float4 p0 = live ? src.plane(0) : make_float4(0.f, 0.f, 0.f, 0.f);
  Fwd f;
  bool intrinsics = false;
  for (int b = 0; b < pv.batch; ++b) {
    const Cam& k = pv.k[b];
    bool visible = false;
    if (live) {
      const float pz = k.R[6] * p0.x + k.R[7] * p0.y + k.R[8] * p0.z + k.t[2];
      if (pz > k.znear) {  // the near-plane cull needs only the mean
        if (!intrinsics) {
          project_intrinsics(src, f);
          // the SH planes once per Gaussian, not once per visible view
#pragma unroll
          for (int pl = 0; pl < 12; ++pl) sh[pl * kProjThreads + t] = ldg4(params, (int64_t)(3 + pl) * n + i);
          intrinsics = true;
        }
        visible = project_view(src, k, f);
      }
      if (visible) emit_projection(staged, f, pv.campos[b], pv.proj[b], n, i);
      else emit_culled(pv.proj[b], n, i);
    }
    if (pv.bits) {  // 32 consecutive Gaussians per warp: one bitset word per view
      const uint32_t m = __ballot_sync(0xffffffffu, visible);
      if ((t & 31) == 0 && (i >> 5) < pv.bits_words) pv.bits[b * pv.bits_stride + (i >> 5)] = m;
    }
  }
}

// Reverse mode of the projection of Gaussian i for one camera: parameter gradients from its
// screen-space gradients g0 = (du, dv, dopacity), g1 = (dA, dB, dC), g2 = (dr, dg, db).
// The SH-coefficient gradient is rank one, gcol[c] * y[k] for coefficient k and channel c,
// so it is returned as the clamped colour gradient gcol and the basis y.
struct BwdOut {
  float gm[3];     // mean
  float glogit;    // opacity logit
  float gls[3];    // log-scales
  float4 gq;       // quaternion (unnormalised)
  float gcol[3];   // colour gradient after the clamp at 0
  SHBasis b;       // SH basis at the view direction
};

template <class Src>
__device__ __forceinline__ void project_bwd_core(const Src& src, const Cam& k, float3 campos, const Fwd& f, float4 g0,
                                                 float4 g1, float4 g2, BwdOut& o) {
  const float4 p0 = src.plane(0);

  // ---- colour: rgb = max(sum_k sh_k Y_k(d) + 0.5, 0), d = (mean - campos)/|.|
  float dx = p0.x - campos.x, dy = p0.y - campos.y, dz = p0.z - campos.z;
  const float il = rsqrtf(dx * dx + dy * dy + dz * dz);
  dx *= il; dy *= il; dz *= il;
  sh_eval(dx, dy, dz, o.b);
  float sh[48];
#pragma unroll
  for (int pl = 0; pl < 12; ++pl) {
    const float4 s = src.plane(3 + pl);
    sh[4 * pl + 0] = s.x; sh[4 * pl + 1] = s.y; sh[4 * pl + 2] = s.z; sh[4 * pl + 3] = s.w;
  }
  o.gcol[0] = g2.x; o.gcol[1] = g2.y; o.gcol[2] = g2.z;
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    float raw = 0.5f;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) raw += sh[3 * kk + c] * o.b.y[kk];
    if (raw < 0.f) o.gcol[c] = 0.f;  // clamped channel passes no gradient
  }
  float wsum[16];
#pragma unroll
  for (int kk = 0; kk < 16; ++kk)
    wsum[kk] = o.gcol[0] * sh[3 * kk] + o.gcol[1] * sh[3 * kk + 1] + o.gcol[2] * sh[3 * kk + 2];
  const float3 gd = sh_grad_dot(dx, dy, dz, wsum);
  const float gdot = gd.x * dx + gd.y * dy + gd.z * dz;
  float gmx = (gd.x - gdot * dx) * il, gmy = (gd.y - gdot * dy) * il, gmz = (gd.z - gdot * dz) * il;

  // ---- conic = inverse of the dilated covariance: dL/dcov = -Q G Q (symmetric form)
  const float gA = g1.x, gBh = 0.5f * g1.y, gC = g1.z;
  const float qg00 = f.A * gA + f.B * gBh, qg01 = f.A * gBh + f.B * gC;
  const float qg10 = f.B * gA + f.C * gBh, qg11 = f.B * gBh + f.C * gC;
  const float D00 = -(qg00 * f.A + qg01 * f.B);
  const float D01 = -(qg00 * f.B + qg01 * f.C);
  const float D11 = -(qg10 * f.B + qg11 * f.C);
  // ---- cov = Tm Sigma Tm^T:  dSigma = Tm^T D Tm,  dTm = 2 D Tm Sigma
  const float* T0 = f.T0;
  const float* T1 = f.T1;
  float dS[6];
  {
    float v0[3], v1[3];  // D Tm rows
#pragma unroll
    for (int c = 0; c < 3; ++c) {
      v0[c] = D00 * T0[c] + D01 * T1[c];
      v1[c] = D01 * T0[c] + D11 * T1[c];
    }
    dS[0] = T0[0] * v0[0] + T1[0] * v1[0];
    dS[1] = T0[0] * v0[1] + T1[0] * v1[1];
    dS[2] = T0[0] * v0[2] + T1[0] * v1[2];
    dS[3] = T0[1] * v0[1] + T1[1] * v1[1];
    dS[4] = T0[1] * v0[2] + T1[1] * v1[2];
    dS[5] = T0[2] * v0[2] + T1[2] * v1[2];
    const float* S = f.Sg;
    float dT0[3], dT1[3];
    dT0[0] = 2.f * (v0[0] * S[0] + v0[1] * S[1] + v0[2] * S[2]);
    dT0[1] = 2.f * (v0[0] * S[1] + v0[1] * S[3] + v0[2] * S[4]);
    dT0[2] = 2.f * (v0[0] * S[2] + v0[1] * S[4] + v0[2] * S[5]);
    dT1[0] = 2.f * (v1[0] * S[0] + v1[1] * S[1] + v1[2] * S[2]);
    dT1[1] = 2.f * (v1[0] * S[1] + v1[1] * S[3] + v1[2] * S[4]);
    dT1[2] = 2.f * (v1[0] * S[2] + v1[1] * S[4] + v1[2] * S[5]);
    // Tm = J W: only J00, J02, J11, J12 are variable
    const float dJ00 = dT0[0] * k.R[0] + dT0[1] * k.R[1] + dT0[2] * k.R[2];
    const float dJ02 = dT0[0] * k.R[6] + dT0[1] * k.R[7] + dT0[2] * k.R[8];
    const float dJ11 = dT1[0] * k.R[3] + dT1[1] * k.R[4] + dT1[2] * k.R[5];
    const float dJ12 = dT1[0] * k.R[6] + dT1[1] * k.R[7] + dT1[2] * k.R[8];
    const float iz = 1.f / f.pz, iz2 = iz * iz;
    float gpx = g0.x * k.fx * iz;
    float gpy = g0.y * k.fy * iz;
    float gpz = -(g0.x * k.fx * f.px + g0.y * k.fy * f.py) * iz2;
    gpz += -(dJ00 * k.fx + dJ11 * k.fy) * iz2;
    if (f.clx) {
      gpz += dJ02 * k.fx * f.xr * iz2;
    } else {
      gpx += -dJ02 * k.fx * iz2;
      gpz += 2.f * dJ02 * k.fx * f.px * iz2 * iz;
    }
    if (f.cly) {
      gpz += dJ12 * k.fy * f.yr * iz2;
    } else {
      gpy += -dJ12 * k.fy * iz2;
      gpz += 2.f * dJ12 * k.fy * f.py * iz2 * iz;
    }
    // p_cam = W mean + t
    gmx += k.R[0] * gpx + k.R[3] * gpy + k.R[6] * gpz;
    gmy += k.R[1] * gpx + k.R[4] * gpy + k.R[7] * gpz;
    gmz += k.R[2] * gpx + k.R[5] * gpy + k.R[8] * gpz;
  }
  o.gm[0] = gmx; o.gm[1] = gmy; o.gm[2] = gmz;
  // ---- Sigma = M M^T, M = Rq diag(s):  dM = 2 dSigma M
  float M[9];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int c = 0; c < 3; ++c) M[3 * r + c] = f.Rq[3 * r + c] * f.s[c];
  const float dSf[9] = {dS[0], dS[1], dS[2], dS[1], dS[3], dS[4], dS[2], dS[4], dS[5]};
  float dM[9];
#pragma unroll
  for (int r = 0; r < 3; ++r)
#pragma unroll
    for (int c = 0; c < 3; ++c)
      dM[3 * r + c] = 2.f * (dSf[3 * r] * M[c] + dSf[3 * r + 1] * M[3 + c] + dSf[3 * r + 2] * M[6 + c]);
  float dR[9];
#pragma unroll
  for (int c = 0; c < 3; ++c) {
    o.gls[c] = (dM[c] * f.Rq[c] + dM[3 + c] * f.Rq[3 + c] + dM[6 + c] * f.Rq[6 + c]) * f.s[c];
#pragma unroll
    for (int r = 0; r < 3; ++r) dR[3 * r + c] = dM[3 * r + c] * f.s[c];
  }
  // ---- rotation matrix of the normalised quaternion (w, x, y, z)
  const float w = f.qn[0], x = f.qn[1], y = f.qn[2], z = f.qn[3];
  float gq[4];
  gq[0] = 2.f * (z * (dR[3] - dR[1]) + y * (dR[2] - dR[6]) + x * (dR[7] - dR[5]));
  gq[1] = 2.f * (y * (dR[1] + dR[3]) + z * (dR[2] + dR[6]) + w * (dR[7] - dR[5]) - 2.f * x * (dR[4] + dR[8]));
  gq[2] = 2.f * (x * (dR[1] + dR[3]) + w * (dR[2] - dR[6]) + z * (dR[5] + dR[7]) - 2.f * y * (dR[0] + dR[8]));
  gq[3] = 2.f * (w * (dR[3] - dR[1]) + x * (dR[2] + dR[6]) + y * (dR[5] + dR[7]) - 2.f * z * (dR[0] + dR[4]));
  const float qd = gq[0] * w + gq[1] * x + gq[2] * y + gq[3] * z;
  o.gq = make_float4((gq[0] - qd * w) * f.qinv, (gq[1] - qd * x) * f.qinv, (gq[2] - qd * y) * f.qinv,
                     (gq[3] - qd * z) * f.qinv);
  // ---- opacity = sigmoid(logit)
  o.glogit = g0.z * f.opac * (1.f - f.opac);
}

__global__ void __launch_bounds__(256) k_project_bwd(const float* __restrict__ params, int64_t n, Cam k,
                                                     float3 campos, const float* __restrict__ proj,
                                                     const float* __restrict__ grad2d, float* __restrict__ grads,
                                                     float2* __restrict__ stat) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (__float_as_int(ldg4(proj, n + i).w) <= 0) return;  // culled in this view
  Fwd f;
  const GlobalParams src{params, n, i};
  if (!project_core(src, k, f)) return;
  BwdOut o;
  const float4 g0 = ldg4(grad2d, 3 * i + 0);
  project_bwd_core(src, k, campos, f, g0, ldg4(grad2d, 3 * i + 1), ldg4(grad2d, 3 * i + 2), o);
  if (stat) {  // densification statistic: this view's screen-space mean-gradient length
    float2 s2 = stat[i];
    s2.x += sqrtf(g0.x * g0.x + g0.y * g0.y);
    s2.y += 1.f;
    stat[i] = s2;
  }
  // ---- accumulate into the gradient planes
  float4* G = reinterpret_cast<float4*>(grads);
  float4 a0 = G[i];
  a0.x += o.gm[0]; a0.y += o.gm[1]; a0.z += o.gm[2]; a0.w += o.glogit;
  G[i] = a0;
  float4 a1 = G[n + i];
  a1.x += o.gls[0]; a1.y += o.gls[1]; a1.z += o.gls[2];
  G[n + i] = a1;
  float4 a2 = G[2 * n + i];
  a2.x += o.gq.x; a2.y += o.gq.y; a2.z += o.gq.z; a2.w += o.gq.w;
  G[2 * n + i] = a2;
#pragma unroll
  for (int pl = 0; pl < 12; ++pl) {
    float4 s = G[(int64_t)(3 + pl) * n + i];
    float* sv = reinterpret_cast<float*>(&s);
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      const int fidx = 4 * pl + l;
      sv[l] += o.gcol[fidx % 3] * o.b.y[fidx / 3];
    }
    G[(int64_t)(3 + pl) * n + i] = s;
  }
}

// ------------------------------------------------------------------ batched backward + Adam
// The composition of gs_project_bwd over the views of a batch (gradients summed in view
// order) and gs_sparse_adam over the Gaussians visible in at least one of them, without the
// gradient planes ever reaching global memory: a thread owns one Gaussian, keeps its
// geometry gradients in registers and its 48 SH-coefficient gradients in shared memory, and
// applies the update plane by plane.  Reads 240 B of parameters + 64 B per view + 480 B of
// moments and writes 720 B per updated Gaussian.
constexpr int kMaxBatchViews = 16;
constexpr int kAdamThreads = 128;

struct BatchViews {
  Cam k[kMaxBatchViews];
  float3 campos[kMaxBatchViews];
  const float* proj[kMaxBatchViews];
  const float* grad2d[kMaxBatchViews];
  const uint32_t* bits;  // optional visibility bitsets [batch][bits_stride]
  int64_t bits_stride;
  int batch;
};

struct AdamHyper {
  float b1, b2, eps;
  float lr_c;    // lr sqrt(batch) / (1 - beta1'^step): the step size with the first bias correction
  float ibc2;    // 1 / (1 - beta2'^step)
};

__device__ __forceinline__ void adam4(float4& p, float4& m, float4& v, float4 g, const AdamHyper& h) {
  float* pa = &p.x;
  float* ma = &m.x;
  float* va = &v.x;
  const float ga[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
  for (int l = 0; l < 4; ++l) {
    ma[l] = h.b1 * ma[l] + (1.f - h.b1) * ga[l];
    va[l] = h.b2 * va[l] + (1.f - h.b2) * ga[l] * ga[l];
    // the bias corrections as host-computed factors, one fast division: a few ulp of the
    // update, far inside its tolerance, instead of two IEEE divisions per element
    pa[l] -= __fdividef(h.lr_c * ma[l], sqrtf(va[l] * h.ibc2) + h.eps);
  }
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

struct AdamSmem {
  float4 par[15][kAdamThreads];  // the CTA's parameter planes
  float4 sh[12][kAdamThreads];   // SH-coefficient gradients in the planes' layout: [q][thread] holds
                                 // coefficients 3k + c = 4q .. 4q + 3 (one 16-byte access per four)
};

__global__ void __launch_bounds__(kAdamThreads, 4) k_project_bwd_adam(float* __restrict__ params, int64_t n,
                                                                      BatchViews bv, float4* __restrict__ m,
                                                                      float4* __restrict__ v, AdamHyper h,
                                                                      const int64_t* counts, int n_counts,
                                                                      float2* __restrict__ stat) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  AdamSmem& S = *reinterpret_cast<AdamSmem*>(smem_raw);
  for (int c = 0; c < n_counts; ++c)
    if (counts[2 * c + 1] != 0) return;  // a view of this batch overflowed its binning
  const int t = threadIdx.x;
  const int64_t i = (int64_t)blockIdx.x * kAdamThreads + t;
  if (i >= n) return;
  // the fifteen planes of this Gaussian, copied asynchronously while the visibility is read
  const float4* P4 = reinterpret_cast<const float4*>(params);
#pragma unroll
  for (int pl = 0; pl < 15; ++pl) cp_async16(&S.par[pl][t], &P4[(int64_t)pl * n + i]);
  asm volatile("cp.async.commit_group;" ::: "memory");
  float4 (*s_sh)[kAdamThreads] = S.sh;
#pragma unroll
  for (int q = 0; q < 12; ++q) s_sh[q][t] = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 ga = make_float4(0.f, 0.f, 0.f, 0.f), gl = ga, gq = ga;
  bool seen = false;
  float dsum = 0.f, dcnt = 0.f;  // densification statistic of the batch's views
  uint32_t vis = 0;  // views whose radius word is > 0 (or visibility bit), all read up front
  if (bv.bits) {
    for (int b = 0; b < bv.batch; ++b)
      vis |= ((__ldg(&bv.bits[b * bv.bits_stride + (i >> 5)]) >> (i & 31)) & 1u) << b;
  } else {
    for (int b = 0; b < bv.batch; ++b)
      if (__float_as_int(__ldg(&reinterpret_cast<const float4*>(bv.proj[b])[n + i].w)) > 0) vis |= 1u << b;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // own copies only: no block barrier needed
  const SharedParams<kAdamThreads> src{&S.par[0][0], t};
  for (int b = 0; b < bv.batch; ++b) {
    if (!((vis >> b) & 1u)) continue;  // culled in this view
    const float* g2 = bv.grad2d[b];
    const float4 g0 = ldg4(g2, 3 * i + 0), g1 = ldg4(g2, 3 * i + 1), g2v = ldg4(g2, 3 * i + 2);
    // the view-independent part is recomputed per view: keeping it live across the views
    // costs more in spilled registers than it saves
    Fwd f;
    if (!project_core(src, bv.k[b], f)) continue;
    seen = true;
    dsum += sqrtf(g0.x * g0.x + g0.y * g0.y);
    dcnt += 1.f;
    BwdOut o;
    project_bwd_core(src, bv.k[b], bv.campos[b], f, g0, g1, g2v, o);
    ga.x += o.gm[0]; ga.y += o.gm[1]; ga.z += o.gm[2]; ga.w += o.glogit;
    gl.x += o.gls[0]; gl.y += o.gls[1]; gl.z += o.gls[2];
    gq.x += o.gq.x; gq.y += o.gq.y; gq.z += o.gq.z; gq.w += o.gq.w;
#pragma unroll
    for (int q = 0; q < 12; ++q) {
      float4 a = s_sh[q][t];
      a.x += o.gcol[(4 * q) % 3] * o.b.y[(4 * q) / 3];
      a.y += o.gcol[(4 * q + 1) % 3] * o.b.y[(4 * q + 1) / 3];
      a.z += o.gcol[(4 * q + 2) % 3] * o.b.y[(4 * q + 2) / 3];
      a.w += o.gcol[(4 * q + 3) % 3] * o.b.y[(4 * q + 3) / 3];
      s_sh[q][t] = a;
    }
  }
  if (!seen) return;  // not visible in any view of the batch: untouched
  if (stat) {
    float2 s2 = stat[i];
    s2.x += dsum;
    s2.y += dcnt;
    stat[i] = s2;
  }
  float4* P = reinterpret_cast<float4*>(params);
  // planes in groups of three: the six moment loads of a group are in flight together
#pragma unroll 1
  for (int pl0 = 0; pl0 < 15; pl0 += 3) {
    float4 pp[3], mm[3], vv[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int64_t e = (int64_t)(pl0 + j) * n + i;
      pp[j] = S.par[pl0 + j][t];
      mm[j] = m[e];
      vv[j] = v[e];
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int pl = pl0 + j;
      float4 g;
      if (pl == 0) g = ga;
      else if (pl == 1) g = gl;
      else if (pl == 2) g = gq;
      else g = s_sh[pl - 3][t];
      adam4(pp[j], mm[j], vv[j], g, h);
      const int64_t e = (int64_t)pl * n + i;
      P[e] = pp[j];
      m[e] = mm[j];
      v[e] = vv[j];
    }
  }
}

float3 camera_centre(const gs_camera& c) {
  // centre = -R^T t
  return make_float3(-(c.R[0] * c.t[0] + c.R[3] * c.t[1] + c.R[6] * c.t[2]),
                     -(c.R[1] * c.t[0] + c.R[4] * c.t[1] + c.R[7] * c.t[2]),
                     -(c.R[2] * c.t[0] + c.R[5] * c.t[1] + c.R[8] * c.t[2]));
}

}  // namespace

extern "C" gs_status gs_project(const float* params, int64_t n, const gs_camera* cam, float* proj, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_project: bad n %lld", (long long)n);
  if (n == 0) return GS_OK;
  if (!params || !proj) return gs::set_error(GS_ERR_INVALID, "gs_project: NULL pointer");
  if (!gs::aligned16(params) || !gs::aligned16(proj))
    return gs::set_error(GS_ERR_INVALID, "gs_project: params/proj must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const int threads = 256;
  const unsigned blocks = (unsigned)((n + threads - 1) / threads);
  k_project_fwd<<<blocks, threads, 0, gs::as_stream(stream)>>>(params, n, k, camera_centre(*cam), proj);
  return gs::check_launch("gs_project");
}

extern "C" gs_status gs_project_batch(const float* params, int64_t n, const gs_camera* cams, int batch,
                                      float* const* projs, uint32_t* visible_bits, int64_t bits_stride,
                                      void* stream) {
  if (batch < 1) return gs::set_error(GS_ERR_INVALID, "gs_project_batch: batch must be >= 1");
  if (n < 0 || n > (int64_t(1) << 31))
    return gs::set_error(GS_ERR_INVALID, "gs_project_batch: bad n %lld", (long long)n);
  if (!cams || !projs) return gs::set_error(GS_ERR_INVALID, "gs_project_batch: NULL pointer");
  for (int b = 0; b < batch; ++b) {
    if (gs_status s = gs::check_camera(&cams[b])) return s;
    if (n > 0 && (!projs[b] || !gs::aligned16(projs[b])))
      return gs::set_error(GS_ERR_INVALID, "gs_project_batch: view %d proj NULL or misaligned", b);
  }
  if (n == 0) return GS_OK;
  if (!params || !gs::aligned16(params))
    return gs::set_error(GS_ERR_INVALID, "gs_project_batch: params NULL or misaligned");
  if (visible_bits && bits_stride < (n + 31) / 32)
    return gs::set_error(GS_ERR_INVALID, "gs_project_batch: bits_stride %lld < ceil(n / 32)", (long long)bits_stride);
  const unsigned blocks = (unsigned)((n + kProjThreads - 1) / kProjThreads);
  const int smem = (int)(12 * kProjThreads * sizeof(float4));
  const cudaError_t attr = gs::max_dynamic_smem((const void*)k_project_fwd_batch, smem);
  if (attr != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_project_batch: %s", cudaGetErrorString(attr));
  for (int b0 = 0; b0 < batch; b0 += kMaxProjViews) {
    ProjViews pv{};
    pv.batch = std::min(kMaxProjViews, batch - b0);
    pv.bits = visible_bits ? visible_bits + (int64_t)b0 * bits_stride : nullptr;
    pv.bits_stride = bits_stride;
    pv.bits_words = (n + 31) / 32;
    for (int b = 0; b < pv.batch; ++b) {
      pv.k[b] = gs::make_cam(cams[b0 + b]);
      pv.campos[b] = camera_centre(cams[b0 + b]);
      pv.proj[b] = projs[b0 + b];
    }
    k_project_fwd_batch<<<blocks, kProjThreads, smem, gs::as_stream(stream)>>>(params, n, pv);
    if (gs_status s = gs::check_launch("gs_project_batch")) return s;
  }
  return GS_OK;
}

extern "C" gs_status gs_project_bwd(const float* params, int64_t n, const gs_camera* cam, const float* proj,
                                    const float* grad2d, float* grads, float* densify_stat, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_project_bwd: bad n");
  if (n == 0) return GS_OK;
  if (!params || !proj || !grad2d || !grads) return gs::set_error(GS_ERR_INVALID, "gs_project_bwd: NULL pointer");
  if (!gs::aligned16(params) || !gs::aligned16(proj) || !gs::aligned16(grad2d) || !gs::aligned16(grads))
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd: arrays must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const int threads = 256;
  const unsigned blocks = (unsigned)((n + threads - 1) / threads);
  if (densify_stat && !gs::aligned8(densify_stat))
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd: densify_stat must be 8-byte aligned");
  k_project_bwd<<<blocks, threads, 0, gs::as_stream(stream)>>>(params, n, k, camera_centre(*cam), proj, grad2d,
                                                               grads, reinterpret_cast<float2*>(densify_stat));
  return gs::check_launch("gs_project_bwd");
}

extern "C" gs_status gs_project_bwd_adam(float* params, int64_t n, const gs_camera* cams, int batch,
                                         const float* const* proj_per_view, const float* const* grad2d_per_view,
                                         float* exp_avg, float* exp_avg_sq, float lr, float beta1, float beta2,
                                         float eps, int64_t step, const int64_t* counts, int n_counts,
                                         float* densify_stat, const uint32_t* visible_bits, int64_t bits_stride,
                                         void* stream) {
  if (batch < 1 || batch > kMaxBatchViews)
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: batch must be 1..%d", kMaxBatchViews);
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: bad n");
  if (step < 1) return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: step must be >= 1");
  if (!cams || !proj_per_view || !grad2d_per_view)
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: NULL pointer");
  if (n == 0) return GS_OK;
  if (!params || !exp_avg || !exp_avg_sq || (n_counts > 0 && !counts))
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: NULL pointer");
  if (n_counts < 0 || !counts) n_counts = 0;
  if (!gs::aligned16(params) || !gs::aligned16(exp_avg) || !gs::aligned16(exp_avg_sq))
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: planes must be 16-byte aligned");
  if (visible_bits && bits_stride < (n + 31) / 32)
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: bits_stride %lld < ceil(n / 32)", (long long)bits_stride);
  BatchViews bv{};
  bv.batch = batch;
  bv.bits = visible_bits;
  bv.bits_stride = bits_stride;
  for (int b = 0; b < batch; ++b) {
    if (gs_status s = gs::check_camera(&cams[b])) return s;
    if (!proj_per_view[b] || !grad2d_per_view[b] || !gs::aligned16(proj_per_view[b]) ||
        !gs::aligned16(grad2d_per_view[b]))
      return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: view %d proj/grad2d NULL or misaligned", b);
    bv.k[b] = gs::make_cam(cams[b]);
    bv.campos[b] = camera_centre(cams[b]);
    bv.proj[b] = proj_per_view[b];
    bv.grad2d[b] = grad2d_per_view[b];
  }
  // batch scaling rule: lr sqrt(b), beta^b; bias corrections with the scaled betas
  const double b1 = std::pow((double)beta1, batch), b2 = std::pow((double)beta2, batch);
  const double lr_b = (double)lr * std::sqrt((double)batch);
  const double bc1 = 1.0 - std::pow(b1, (double)step), bc2 = 1.0 - std::pow(b2, (double)step);
  const AdamHyper h{(float)b1, (float)b2, eps, (float)(lr_b / bc1), (float)(1.0 / bc2)};
  const unsigned blocks = (unsigned)((n + kAdamThreads - 1) / kAdamThreads);
  const cudaError_t attr = gs::max_dynamic_smem((const void*)k_project_bwd_adam, (int)sizeof(AdamSmem));
  if (attr != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_project_bwd_adam: %s", cudaGetErrorString(attr));
  if (densify_stat && !gs::aligned8(densify_stat))
    return gs::set_error(GS_ERR_INVALID, "gs_project_bwd_adam: densify_stat must be 8-byte aligned");
  k_project_bwd_adam<<<blocks, kAdamThreads, sizeof(AdamSmem), gs::as_stream(stream)>>>(
      params, n, bv, reinterpret_cast<float4*>(exp_avg), reinterpret_cast<float4*>(exp_avg_sq), h, counts, n_counts,
      reinterpret_cast<float2*>(densify_stat));
  return gs::check_launch("gs_project_bwd_adam");
}
