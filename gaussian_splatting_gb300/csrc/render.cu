// Per-tile alpha compositing (gs_render_fwd) and its reverse-order backward (gs_render_bwd).
//
// One CTA per 16x16 tile, one thread per pixel.  The tile's depth-sorted list is walked in
// batches of 256 Gaussians: each thread gathers one Gaussian's screen-space record into
// shared memory, then every pixel evaluates the whole batch from shared memory (broadcast
// reads).  A CTA stops fetching batches once every pixel has saturated
// (__syncthreads_count).  The conic is pre-scaled by log2(e) so alpha = opacity * 2^p is
// one ex2 on the special-function unit; forward and backward evaluate alpha through the
// same function so the backward's T / (1 - alpha) recovery retraces the forward exactly.
#include "common.cuh"

namespace {

constexpr int kBatch = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kAlphaMax = 0.99f;
constexpr float kTMin = 1e-4f;

// Gathered record: s0 = (u, v, a2, b2), s1 = (c2, opacity, r, g), s2 = b, where
// (a2, b2, c2) = log2(e) * (-A/2, -B, -C/2) so that p = a2 dx^2 + b2 dx dy + c2 dy^2
// = log2(e) * power.
__device__ __forceinline__ void gather_record(const float* __restrict__ proj, int64_t n, uint32_t g, float4& s0,
                                              float4& s1, float& s2) {
  const float4 q0 = ldg4(proj, g);
  const float4 q1 = ldg4(proj, n + g);
  const float4 q2 = ldg4(proj, 2 * n + g);
  s0 = make_float4(q0.x, q0.y, -0.5f * kLog2e * q1.x, -kLog2e * q1.y);
  s1 = make_float4(-0.5f * kLog2e * q1.z, q0.w, q2.x, q2.y);
  s2 = q2.z;
}

// p (log2 units) at pixel-centre offset (dx, dy) = centre - (u, v).  Written with explicit
// roundings so that the forward and backward kernels evaluate the same bits.
__device__ __forceinline__ float power2(const float4& s0, const float4& s1, float dx, float dy) {
  const float t = fmaf(s0.w, dy, __fmul_rn(s0.z, dx));
  return fmaf(__fmul_rn(s1.x, dy), dy, __fmul_rn(dx, t));
}

__device__ __forceinline__ float alpha_of(float opacity, float G) {
  return fminf(kAlphaMax, __fmul_rn(opacity, G));
}

__global__ void __launch_bounds__(256) k_render_fwd(const float* __restrict__ proj, int64_t n,
                                                    const uint32_t* __restrict__ vals,
                                                    const uint32_t* __restrict__ ranges, int W, int H, int Tx,
                                                    float3 bg, float* __restrict__ image, float* __restrict__ T_final,
                                                    uint32_t* __restrict__ n_contrib) {
  __shared__ float4 s0[kBatch];
  __shared__ float4 s1[kBatch];
  __shared__ float s2[kBatch];
  const int tile = blockIdx.x;
  const int tx = tile % Tx, ty = tile / Tx;
  const int px = tx * gs::kTile + (threadIdx.x & 15), py = ty * gs::kTile + (threadIdx.x >> 4);
  const bool inside = px < W && py < H;
  const float fx = (float)px + 0.5f, fy = (float)py + 0.5f;
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  float T = 1.f, cr = 0.f, cg = 0.f, cb = 0.f;
  uint32_t last = 0;
  bool done = !inside;
  for (uint32_t b0 = start; b0 < end; b0 += kBatch) {
    if (__syncthreads_count(done) == (int)blockDim.x) break;
    const uint32_t j = b0 + threadIdx.x;
    if (j < end) {
      float4 a, c;
      float d;
      gather_record(proj, n, __ldg(&vals[j]), a, c, d);
      s0[threadIdx.x] = a;
      s1[threadIdx.x] = c;
      s2[threadIdx.x] = d;
    }
    __syncthreads();
    const int cnt = (int)min((uint32_t)kBatch, end - b0);
    for (int k = 0; k < cnt && !done; ++k) {
      const float4 a = s0[k];
      const float4 c = s1[k];
      const float dx = fx - a.x, dy = fy - a.y;
      const float p = power2(a, c, dx, dy);
      if (p > 0.f) continue;
      const float alpha = alpha_of(c.y, fast_exp2(p));
      if (alpha < kAlphaMin) continue;
      const float Tn = __fmul_rn(T, __fsub_rn(1.f, alpha));
      if (Tn < kTMin) {
        done = true;
        break;
      }
      const float w = alpha * T;
      cr = fmaf(w, c.z, cr);
      cg = fmaf(w, c.w, cg);
      cb = fmaf(w, s2[k], cb);
      T = Tn;
      last = b0 - start + (uint32_t)k + 1u;
    }
    __syncthreads();
  }
  if (inside) {
    const int64_t pix = (int64_t)py * W + px;
    const int64_t P = (int64_t)W * H;
    image[pix] = cr + T * bg.x;
    image[P + pix] = cg + T * bg.y;
    image[2 * P + pix] = cb + T * bg.z;
    T_final[pix] = T;
    n_contrib[pix] = last;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(256) k_render_bwd(const float* __restrict__ proj, int64_t n,
                                                    const uint32_t* __restrict__ vals,
                                                    const uint32_t* __restrict__ ranges, int W, int H, int Tx,
                                                    float3 bg, const float* __restrict__ T_final,
                                                    const uint32_t* __restrict__ n_contrib,
                                                    const float* __restrict__ dimg, float* __restrict__ grad2d) {
  __shared__ float4 s0[kBatch];
  __shared__ float4 s1[kBatch];
  __shared__ float s2[kBatch];
  __shared__ uint32_t s_g[kBatch];
  __shared__ uint32_t s_max_last;
  const int tile = blockIdx.x;
  const int tx = tile % Tx, ty = tile / Tx;
  const int px = tx * gs::kTile + (threadIdx.x & 15), py = ty * gs::kTile + (threadIdx.x >> 4);
  const bool inside = px < W && py < H;
  const float fx = (float)px + 0.5f, fy = (float)py + 0.5f;
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  const int64_t pix = (int64_t)py * W + px;
  const int64_t P = (int64_t)W * H;
  float T = 1.f, dr = 0.f, dg = 0.f, db = 0.f;
  uint32_t last = 0;
  if (inside) {
    T = T_final[pix];
    last = n_contrib[pix];
    dr = dimg[pix];
    dg = dimg[P + pix];
    db = dimg[2 * P + pix];
  }
  // colour composited behind the current entry, starting with the background
  float Sr = T * bg.x, Sg = T * bg.y, Sb = T * bg.z;
  if (threadIdx.x == 0) s_max_last = 0;
  __syncthreads();
  if (last) atomicMax(&s_max_last, last);
  __syncthreads();
  const uint32_t max_last = s_max_last;
  const int lane = threadIdx.x & 31;
  // batches aligned to the list start, walked from the back
  for (int bb = (int)((max_last + kBatch - 1) / kBatch) - 1; bb >= 0; --bb) {
    const uint32_t b0 = start + (uint32_t)bb * kBatch;
    const uint32_t j = b0 + threadIdx.x;
    __syncthreads();
    if (j < end) {
      const uint32_t g = __ldg(&vals[j]);
      float4 a, c;
      float d;
      gather_record(proj, n, g, a, c, d);
      s0[threadIdx.x] = a;
      s1[threadIdx.x] = c;
      s2[threadIdx.x] = d;
      s_g[threadIdx.x] = g;
    }
    __syncthreads();
    const int cnt = (int)min((uint32_t)kBatch, end - b0);
    for (int k = cnt - 1; k >= 0; --k) {
      const uint32_t pos = (uint32_t)bb * kBatch + (uint32_t)k;  // list position
      bool use = pos < last;
      float gu = 0.f, gv = 0.f, go = 0.f, gA = 0.f, gB = 0.f, gC = 0.f, gr = 0.f, gg = 0.f, gbl = 0.f;
      float4 a, c;
      if (__any_sync(0xffffffffu, use)) {
        a = s0[k];
        c = s1[k];
        float dx = 0.f, dy = 0.f, G = 0.f, alpha = 0.f;
        if (use) {
          dx = fx - a.x;
          dy = fy - a.y;
          const float p = power2(a, c, dx, dy);
          G = fast_exp2(p);
          alpha = alpha_of(c.y, G);
          use = !(p > 0.f) && !(alpha < kAlphaMin);
        }
        if (use) {
          const float blue = s2[k];
          T = __fdiv_rn(T, __fsub_rn(1.f, alpha));
          const float w = alpha * T;
          gr = w * dr;
          gg = w * dg;
          gbl = w * db;
          const float dalpha = T * (c.z * dr + c.w * dg + blue * db) - (Sr * dr + Sg * dg + Sb * db) / (1.f - alpha);
          Sr = fmaf(w, c.z, Sr);
          Sg = fmaf(w, c.w, Sg);
          Sb = fmaf(w, blue, Sb);
          if (__fmul_rn(c.y, G) <= kAlphaMax) {
            go = dalpha * G;
            const float dpow = dalpha * alpha;  // d alpha / d power = alpha
            gA = -0.5f * dpow * dx * dx;
            gB = -dpow * dx * dy;
            gC = -0.5f * dpow * dy * dy;
            // natural conic from the log2-scaled record
            const float A = a.z * (-2.f / kLog2e), B = a.w * (-1.f / kLog2e), C = c.x * (-2.f / kLog2e);
            gu = dpow * (A * dx + B * dy);
            gv = dpow * (B * dx + C * dy);
          }
        }
        if (__any_sync(0xffffffffu, use)) {
          gu = warp_sum(gu);
          gv = warp_sum(gv);
          go = warp_sum(go);
          gA = warp_sum(gA);
          gB = warp_sum(gB);
          gC = warp_sum(gC);
          gr = warp_sum(gr);
          gg = warp_sum(gg);
          gbl = warp_sum(gbl);
          if (lane == 0) {
            float* dst = grad2d + 12 * (int64_t)s_g[k];
            red_add_v4(dst, gu, gv, go, 0.f);
            red_add_v4(dst + 4, gA, gB, gC, 0.f);
            red_add_v4(dst + 8, gr, gg, gbl, 0.f);
          }
        }
      }
    }
  }
}

}  // namespace

extern "C" gs_status gs_render_fwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                                   const gs_camera* cam, const float* bg, float* image, float* T_final,
                                   uint32_t* n_contrib, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: bad n");
  if (!ranges || !image || !T_final || !n_contrib || (n > 0 && (!proj || !vals)))
    return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: NULL pointer");
  if (proj && !gs::aligned16(proj)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: proj must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const float3 b = bg ? make_float3(bg[0], bg[1], bg[2]) : make_float3(0.f, 0.f, 0.f);
  k_render_fwd<<<k.Tx * k.Ty, 256, 0, gs::as_stream(stream)>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, image,
                                                                  T_final, n_contrib);
  return gs::check_launch("gs_render_fwd");
}

extern "C" gs_status gs_render_bwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                                   const gs_camera* cam, const float* bg, const float* T_final,
                                   const uint32_t* n_contrib, const float* dL_dimage, float* grad2d, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_render_bwd: bad n");
  if (!ranges || !T_final || !n_contrib || !dL_dimage || (n > 0 && (!proj || !vals || !grad2d)))
    return gs::set_error(GS_ERR_INVALID, "gs_render_bwd: NULL pointer");
  if ((proj && !gs::aligned16(proj)) || (grad2d && !gs::aligned16(grad2d)))
    return gs::set_error(GS_ERR_INVALID, "gs_render_bwd: proj/grad2d must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const float3 b = bg ? make_float3(bg[0], bg[1], bg[2]) : make_float3(0.f, 0.f, 0.f);
  cudaStream_t st = gs::as_stream(stream);
  if (n > 0 && cudaMemsetAsync(grad2d, 0, sizeof(float) * 12 * (size_t)n, st) != cudaSuccess)
    return gs::check_launch("gs_render_bwd memset");
  k_render_bwd<<<k.Tx * k.Ty, 256, 0, st>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, T_final, n_contrib, dL_dimage,
                                            grad2d);
  return gs::check_launch("gs_render_bwd");
}
