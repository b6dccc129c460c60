// Per-tile alpha compositing (gs_render_fwd) and its reverse-order backward (gs_render_bwd).
//
// "Render" and "backpropagation" steps of the Grendel-GS training flow (训练流程): each
// pixel composites the depth-sorted Gaussians of its 16x16 tile front to back; the backward
// walks the same lists back to front.
//
// Layout: one 64-thread CTA per tile, 4 pixels per thread.  Warp 0 owns rows 0-7 and warp 1
// rows 8-15; lane l owns column l % 16 and the four rows 4 (l / 16) .. +3 of its warp's half,
// so a thread's pixels share dx and a warp covers a compact 16x8 block (a Gaussian that
// misses that block is skipped by the whole warp at once).  The tile's list is walked in
// batches of 256 Gaussians gathered into shared memory (4 per thread) and evaluated from
// shared memory with broadcast reads.  The conic is stored scaled by -log2(e)/2 so that
// alpha = opacity * 2^p costs one ex2; a per-Gaussian threshold p_min = log2(1/(255 opacity))
// rejects pairs below the 1/255 skip before the ex2.  Forward and backward evaluate every
// (pixel, Gaussian) pair through the same functions, so the backward's T / (1 - alpha)
// recovery retraces the forward's decisions exactly.
//
// The backward sums each Gaussian's nine gradient terms over a thread's pixels, then over
// the warp with a transposed butterfly (16 shuffles for 16 lanes of values instead of 45),
// and one warp-wide atomic add puts the nine sums into grad2d.
#include "common.cuh"

namespace {

constexpr int kThreads = 64;   // per tile
constexpr int kPPT = 4;        // pixels per thread
constexpr int kBatch = 256;    // Gaussians per shared-memory batch
constexpr int kPerThreadLoad = kBatch / kThreads;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kAlphaMax = 0.99f;
constexpr float kTMin = 1e-4f;

// Gathered record: s0 = (u, v, a2, b2), s1 = (c2, opacity, p_min, Gaussian index bits),
// s2 = (r, g, b, 0) with (a2, b2, c2) = log2(e) * (-A/2, -B, -C/2), so that
// p = a2 dx^2 + b2 dx dy + c2 dy^2 = log2(e) * power.
struct Rec {
  float4 s0, s1, s2;
};

__device__ __forceinline__ Rec gather_record(const float* __restrict__ proj, int64_t n, uint32_t g) {
  const float4 q0 = ldg4(proj, g);
  const float4 q1 = ldg4(proj, n + g);
  const float4 q2 = ldg4(proj, 2 * n + g);
  Rec r;
  r.s0 = make_float4(q0.x, q0.y, -0.5f * kLog2e * q1.x, -kLog2e * q1.y);
  // alpha < 1/255  <=>  p < log2(1 / (255 opacity))
  float lg;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(q0.w * 255.0f));
  r.s1 = make_float4(-0.5f * kLog2e * q1.z, q0.w, -lg, __uint_as_float(g));
  r.s2 = make_float4(q2.x, q2.y, q2.z, 0.f);
  return r;
}

// p at pixel-centre offset (dx, dy), with e = a2 * dx shared by a thread's column.  Explicit
// roundings: the forward and backward kernels must evaluate identical bits.
__device__ __forceinline__ float power2(const float4& s0, const float4& s1, float dx, float e, float dy) {
  const float t = fmaf(s0.w, dy, e);
  return fmaf(__fmul_rn(s1.x, dy), dy, __fmul_rn(dx, t));
}

__device__ __forceinline__ float alpha_of(float opacity, float G) {
  return fminf(kAlphaMax, __fmul_rn(opacity, G));
}

// p passes the skip tests (power <= 0 and alpha >= 1/255 before the clamp)
__device__ __forceinline__ bool candidate(float p, float pmin) { return p >= pmin && !(p > 0.f); }

__device__ __forceinline__ void pixel_of(int tile, int Tx, int lane, int warp, int& px, int& py0) {
  const int tx = tile % Tx, ty = tile / Tx;
  px = tx * gs::kTile + (lane & 15);
  py0 = ty * gs::kTile + warp * 8 + (lane >> 4) * 4;
}

__global__ void __launch_bounds__(kThreads) k_render_fwd(const float* __restrict__ proj, int64_t n,
                                                         const uint32_t* __restrict__ vals,
                                                         const uint32_t* __restrict__ ranges, int W, int H, int Tx,
                                                         float3 bg, float* __restrict__ image,
                                                         float* __restrict__ T_final, uint32_t* __restrict__ n_contrib,
                                                         uint32_t* __restrict__ work) {
  __shared__ float4 s0[kBatch];
  __shared__ float4 s1[kBatch];
  __shared__ float4 s2[kBatch];
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int px, py0;
  pixel_of(tile, Tx, lane, warp, px, py0);
  const float fx = (float)px + 0.5f;
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  float T[kPPT], cr[kPPT], cg[kPPT], cb[kPPT];
  uint32_t last[kPPT], evald[kPPT], used[kPPT];
  bool done[kPPT];
#pragma unroll
  for (int i = 0; i < kPPT; ++i) {
    T[i] = 1.f;
    cr[i] = cg[i] = cb[i] = 0.f;
    last[i] = evald[i] = used[i] = 0;
    done[i] = !(px < W && py0 + i < H);
  }
  for (uint32_t b0 = start; b0 < end; b0 += kBatch) {
    int mine = 0;
#pragma unroll
    for (int i = 0; i < kPPT; ++i) mine += done[i] ? 1 : 0;
    if (__syncthreads_count(mine == kPPT) == kThreads) break;
#pragma unroll
    for (int r = 0; r < kPerThreadLoad; ++r) {
      const int slot = r * kThreads + threadIdx.x;
      const uint32_t j = b0 + slot;
      if (j < end) {
        const Rec rec = gather_record(proj, n, __ldg(&vals[j]));
        s0[slot] = rec.s0;
        s1[slot] = rec.s1;
        s2[slot] = rec.s2;
      }
    }
    __syncthreads();
    const int cnt = (int)min((uint32_t)kBatch, end - b0);
    for (int k = 0; k < cnt; ++k) {
      bool all_done = true;
#pragma unroll
      for (int i = 0; i < kPPT; ++i) all_done &= done[i];
      if (all_done) break;
      const float4 a = s0[k];
      const float4 c = s1[k];
      const float dx = fx - a.x;
      const float e = __fmul_rn(a.z, dx);
#pragma unroll
      for (int i = 0; i < kPPT; ++i) {
        if (done[i]) continue;
        ++evald[i];
        const float dy = ((float)(py0 + i) + 0.5f) - a.y;
        const float p = power2(a, c, dx, e, dy);
        if (!candidate(p, c.z)) continue;
        const float alpha = alpha_of(c.y, fast_exp2(p));
        if (alpha < kAlphaMin) continue;
        const float Tn = __fmul_rn(T[i], __fsub_rn(1.f, alpha));
        if (Tn < kTMin) {
          done[i] = true;
          continue;
        }
        const float4 col = s2[k];
        const float w = alpha * T[i];
        cr[i] = fmaf(w, col.x, cr[i]);
        cg[i] = fmaf(w, col.y, cg[i]);
        cb[i] = fmaf(w, col.z, cb[i]);
        T[i] = Tn;
        last[i] = b0 - start + (uint32_t)k + 1u;
        ++used[i];
      }
    }
    __syncthreads();
  }
  const int64_t P = (int64_t)W * H;
#pragma unroll
  for (int i = 0; i < kPPT; ++i) {
    const int py = py0 + i;
    if (px < W && py < H) {
      const int64_t pix = (int64_t)py * W + px;
      image[pix] = cr[i] + T[i] * bg.x;
      image[P + pix] = cg[i] + T[i] * bg.y;
      image[2 * P + pix] = cb[i] + T[i] * bg.z;
      T_final[pix] = T[i];
      n_contrib[pix] = last[i];
      if (work) {
        work[pix] = evald[i];
        work[P + pix] = used[i];
      }
    }
  }
}

// Sum of 16 per-lane values over the warp by a transposed butterfly: afterwards lanes 2k and
// 2k+1 hold the warp total of value k.  16 shuffles instead of 16 * 5.
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int level = 0; level < 4; ++level) {
    const int off = 16 >> level;  // 16, 8, 4, 2
    const int half = 8 >> level;  // values kept: 8, 4, 2, 1
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      // give away the half the partner keeps; add the partner's copy of the half kept here
      const float give = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

__global__ void __launch_bounds__(kThreads) k_render_bwd(const float* __restrict__ proj, int64_t n,
                                                         const uint32_t* __restrict__ vals,
                                                         const uint32_t* __restrict__ ranges, int W, int H, int Tx,
                                                         float3 bg, const float* __restrict__ T_final,
                                                         const uint32_t* __restrict__ n_contrib,
                                                         const float* __restrict__ dimg, float* __restrict__ grad2d) {
  __shared__ float4 s0[kBatch];
  __shared__ float4 s1[kBatch];
  __shared__ float4 s2[kBatch];
  __shared__ uint32_t s_max_last;
  const int tile = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int px, py0;
  pixel_of(tile, Tx, lane, warp, px, py0);
  const float fx = (float)px + 0.5f;
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  const int64_t P = (int64_t)W * H;
  float T[kPPT], dr[kPPT], dg[kPPT], db[kPPT], Sr[kPPT], Sg[kPPT], Sb[kPPT];
  uint32_t last[kPPT];
  uint32_t my_max = 0;
#pragma unroll
  for (int i = 0; i < kPPT; ++i) {
    const int py = py0 + i;
    T[i] = 1.f;
    dr[i] = dg[i] = db[i] = 0.f;
    last[i] = 0;
    if (px < W && py < H) {
      const int64_t pix = (int64_t)py * W + px;
      T[i] = T_final[pix];
      last[i] = n_contrib[pix];
      dr[i] = dimg[pix];
      dg[i] = dimg[P + pix];
      db[i] = dimg[2 * P + pix];
    }
    // colour composited behind the current entry, starting with the background
    Sr[i] = T[i] * bg.x;
    Sg[i] = T[i] * bg.y;
    Sb[i] = T[i] * bg.z;
    my_max = max(my_max, last[i]);
  }
  if (threadIdx.x == 0) s_max_last = 0;
  __syncthreads();
  my_max = __reduce_max_sync(0xffffffffu, my_max);
  if (lane == 0) atomicMax(&s_max_last, my_max);
  __syncthreads();
  const uint32_t max_last = s_max_last;
  // batches aligned to the list start, walked from the back
  for (int bb = (int)((max_last + kBatch - 1) / kBatch) - 1; bb >= 0; --bb) {
    const uint32_t b0 = start + (uint32_t)bb * kBatch;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPerThreadLoad; ++r) {
      const int slot = r * kThreads + threadIdx.x;
      const uint32_t j = b0 + slot;
      if (j < end) {
        const Rec rec = gather_record(proj, n, __ldg(&vals[j]));
        s0[slot] = rec.s0;
        s1[slot] = rec.s1;
        s2[slot] = rec.s2;
      }
    }
    __syncthreads();
    const int cnt = (int)min((uint32_t)kBatch, min(end, start + max_last) - b0);
    for (int k = cnt - 1; k >= 0; --k) {
      const uint32_t pos = (uint32_t)bb * kBatch + (uint32_t)k;  // list position
      bool any = false;
#pragma unroll
      for (int i = 0; i < kPPT; ++i) any |= pos < last[i];
      if (!__any_sync(0xffffffffu, any)) continue;
      const float4 a = s0[k];
      const float4 c = s1[k];
      const float dx = fx - a.x;
      const float e = __fmul_rn(a.z, dx);
      // natural conic from the log2-scaled record
      const float A = a.z * (-2.f / kLog2e), B = a.w * (-1.f / kLog2e), C = c.x * (-2.f / kLog2e);
      float acc[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) acc[q] = 0.f;
      bool hit = false;
#pragma unroll
      for (int i = 0; i < kPPT; ++i) {
        if (!(pos < last[i])) continue;
        const float dy = ((float)(py0 + i) + 0.5f) - a.y;
        const float p = power2(a, c, dx, e, dy);
        if (!candidate(p, c.z)) continue;
        const float G = fast_exp2(p);
        const float alpha = alpha_of(c.y, G);
        if (alpha < kAlphaMin) continue;
        hit = true;
        const float4 col = s2[k];
        const float om = __fsub_rn(1.f, alpha);
        T[i] = __fdiv_rn(T[i], om);
        const float w = alpha * T[i];
        acc[8] = fmaf(w, dr[i], acc[8]);
        acc[9] = fmaf(w, dg[i], acc[9]);
        acc[10] = fmaf(w, db[i], acc[10]);
        const float dalpha = T[i] * (col.x * dr[i] + col.y * dg[i] + col.z * db[i]) -
                             (Sr[i] * dr[i] + Sg[i] * dg[i] + Sb[i] * db[i]) / om;
        Sr[i] = fmaf(w, col.x, Sr[i]);
        Sg[i] = fmaf(w, col.y, Sg[i]);
        Sb[i] = fmaf(w, col.z, Sb[i]);
        if (__fmul_rn(c.y, G) <= kAlphaMax) {
          acc[2] = fmaf(dalpha, G, acc[2]);
          const float dpow = dalpha * alpha;  // d alpha / d power = alpha
          acc[4] = fmaf(-0.5f * dpow, dx * dx, acc[4]);
          acc[5] = fmaf(-dpow, dx * dy, acc[5]);
          acc[6] = fmaf(-0.5f * dpow, dy * dy, acc[6]);
          acc[0] = fmaf(dpow, A * dx + B * dy, acc[0]);
          acc[1] = fmaf(dpow, B * dx + C * dy, acc[1]);
        }
      }
      if (!__any_sync(0xffffffffu, hit)) continue;
      const float tot = warp_transpose_sum16(acc, lane);
      // lane 2k holds value k; k = 0..11 is the [12] record (3, 7 and 11 are padding)
      const int k_val = lane >> 1;
      if ((lane & 1) == 0 && k_val < 12 && (k_val & 3) != 3) {
        const uint32_t g = __float_as_uint(c.w);
        atomicAdd(grad2d + 12 * (int64_t)g + k_val, tot);
      }
    }
  }
}

}  // namespace

extern "C" gs_status gs_render_fwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                                   const gs_camera* cam, const float* bg, float* image, float* T_final,
                                   uint32_t* n_contrib, uint32_t* work, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: bad n");
  if (!ranges || !image || !T_final || !n_contrib || (n > 0 && (!proj || !vals)))
    return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: NULL pointer");
  if (proj && !gs::aligned16(proj)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: proj must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const float3 b = bg ? make_float3(bg[0], bg[1], bg[2]) : make_float3(0.f, 0.f, 0.f);
  k_render_fwd<<<k.Tx * k.Ty, kThreads, 0, gs::as_stream(stream)>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, image,
                                                                       T_final, n_contrib, work);
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
  k_render_bwd<<<k.Tx * k.Ty, kThreads, 0, st>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, T_final, n_contrib,
                                                 dL_dimage, grad2d);
  return gs::check_launch("gs_render_bwd");
}
