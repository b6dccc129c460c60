// Per-tile alpha compositing (gs_render_fwd) and its reverse-order backward (gs_render_bwd).
//
// "Render" and "backpropagation" steps of the Grendel-GS training flow (训练流程): each
// pixel composites the depth-sorted Gaussians of its 16x16 tile front to back; the backward
// walks the same lists back to front.
//
// Layout: one 128-thread CTA per tile.  The CTAs take the tiles in the order the caller
// gives (gs_tile_order: heaviest first, so that no long tile starts last and runs alone at
// the end of the launch) or, without one, in index order.  Warp w owns the 8x8 block at
// column band w % 2 and row band w / 2 (a square block meets fewer footprints than a 16x4
// one); lane l owns column l % 8 of the block and its two rows 2 (l / 8) + {0, 1}.  The tile's list is walked in
// batches of 256 Gaussians gathered into shared memory (2 per thread).  While gathering,
// each Gaussian gets a 4-bit mask of the warp blocks that its alpha >= 1/255 ellipse meets
// (a box test, then the exact minimum of the quadratic form over the block, with a rounding
// margin), and every warp compacts the batch, in order, into its own list: a warp never
// evaluates a Gaussian whose alpha is below the skip threshold on all of its pixels.
// Per-pixel results are those of walking the full list.  The per-pixel compositing is
// branch-free: a pixel that does not take an entry gets weight zero and keeps its state.
//
// The conic is stored scaled by -log2(e)/2 so that alpha = opacity * 2^p costs one ex2, and
// a per-Gaussian threshold p_min = log2(1/(255 opacity)) rejects pairs below the 1/255 skip
// before the ex2.  Forward and backward evaluate every (pixel, Gaussian) pair through the
// same functions, so both take the same entries with the same alpha; the backward recovers
// each earlier transmittance as T / (1 - alpha) from the forward's final T.
//
// The backward takes two list entries per iteration: for each, a Gaussian's nine gradient
// terms are summed over a thread's two pixels; then both entries' terms are summed over the
// warp together (a 16-value transposed butterfly, 16 shuffles, and a 2-value one for the two
// blue terms, 5 shuffles, instead of 90 for plain butterflies) and eighteen lanes add the sums
// to grad2d with one warp-wide atomic instruction.
#include "common.cuh"

namespace {

constexpr int kThreads = 128;  // per tile
constexpr int kWarps = kThreads / 32;
constexpr int kPPT = 2;        // pixels per thread
constexpr int kBatch = 256;    // Gaussians per shared-memory batch
constexpr int kPerThreadLoad = kBatch / kThreads;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kAlphaMin = 1.0f / 255.0f;
constexpr float kAlphaMax = 0.99f;
constexpr float kTMin = 1e-4f;

struct __align__(16) BatchSmem {
  float4 s0[kBatch];        // (u, v, a2, b2)
  float4 s1[kBatch];        // (c2, opacity, p_min / 2, Gaussian index bits)
  float4 s2[kBatch];        // (r, g, b, 0)
  uint32_t mask[kBatch];    // warp blocks the Gaussian can reach
  uint8_t list[kWarps][kBatch];
  uint32_t count[kWarps];
};

// (a2, b2, c2) = log2(e) * (-A/2, -B, -C/2), so p = a2 dx^2 + b2 dx dy + c2 dy^2 = log2(e) power.
__device__ __forceinline__ void gather_record(const float* __restrict__ proj, int64_t n, uint32_t g, int tile_x0,
                                              int tile_y0, BatchSmem& S, int slot) {
  const float4 q0 = ldg4(proj, g);
  const float4 q1 = ldg4(proj, n + g);
  const float4 q2 = ldg4(proj, 2 * n + g);
  // alpha < 1/255  <=>  p < log2(1 / (255 opacity))
  float lg;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(q0.w * 255.0f));
  S.s0[slot] = make_float4(q0.x, q0.y, -0.5f * kLog2e * q1.x, -kLog2e * q1.y);
  S.s1[slot] = make_float4(-0.5f * kLog2e * q1.z, q0.w, -0.5f * lg, __uint_as_float(g));
  S.s2[slot] = make_float4(q2.x, q2.y, q2.z, 0.f);
  // bounding box of {d : d^T conic d <= K}, K = 2 ln(255 opacity): half-widths sqrt(K Sigma_xx),
  // sqrt(K Sigma_yy) with Sigma = conic^-1; enlarged so rounding never drops a reachable pair
  uint32_t m = 0;
  // (fast intrinsics: the 0.1 % + 0.05 px box slack and the exact test's margin absorb their
  // few-ulp errors, and culling only ever skips pairs no pixel can accept)
  const float Kr = 2.0f * __logf(255.0f * q0.w);
  const float K = fmaxf(Kr, 0.f);  // opacity at the 1/255 threshold within the log's error: keep it
  const float det = q1.x * q1.z - q1.y * q1.y;
  if (Kr > -1e-5f && det > 0.f) {
    const float idet = __fdividef(1.f, det);
    const float hx = sqrtf(K * q1.z * idet) * 1.001f + 0.05f;
    const float hy = sqrtf(K * q1.x * idet) * 1.001f + 0.05f;
    // Per warp block (8x8 pixels, block w at column band w & 1, row band w >> 1): the box test,
    // then the exact test: the minimum of q(d) = A dx^2 + 2B dx dy + C dy^2 over the block's
    // rectangle of pixel centres (d relative to the mean) against K.  q is convex; its minimum
    // over the column strip [X0, X1] lies at dx = 0 when the strip holds the mean, else on the
    // nearer edge X at dy = -B X / C; clamping that dy to the block's rows and then dx to the
    // columns gives the minimum over the rectangle.  The margin keeps every block whose pixels
    // the fp32 candidate test could accept.
    const float A = q1.x, B = q1.y, C = q1.z;
    const float rBA = -__fdividef(B, A), rBC = -__fdividef(B, C), Kk = K * 1.001f + 1e-3f;
#pragma unroll
    for (int bx = 0; bx < 2; ++bx) {
      const float xmin = (float)(tile_x0 + 8 * bx) + 0.5f, xmax = xmin + 7.0f;
      if (!(q0.x + hx >= xmin && q0.x - hx <= xmax)) continue;
      const float X0 = xmin - q0.x, X1 = xmax - q0.x;
      const float xe = X0 > 0.f ? X0 : (X1 < 0.f ? X1 : 0.f);
      const float dys = rBC * xe;
#pragma unroll
      for (int by = 0; by < 2; ++by) {
        const float ymin = (float)(tile_y0 + 8 * by) + 0.5f, ymax = ymin + 7.0f;
        if (q0.y + hy >= ymin && q0.y - hy <= ymax) {
          const float dy = fminf(fmaxf(dys, ymin - q0.y), ymax - q0.y);
          const float dx = fminf(fmaxf(rBA * dy, X0), X1);
          const float q = A * dx * dx + 2.f * B * dx * dy + C * dy * dy;
          if (q <= Kk) m |= 1u << (bx + 2 * by);
        }
      }
    }
  } else if (!(det > 0.f) && Kr > -1e-5f) {
    m = (1u << kWarps) - 1u;  // degenerate record: keep it everywhere
  }
  S.mask[slot] = m;
}

// Ordered compaction of the batch entries whose mask has this warp's bit.
__device__ __forceinline__ void build_list(BatchSmem& S, int cnt, int warp, int lane) {
  uint32_t total = 0;
  for (int base = 0; base < cnt; base += 32) {
    const int k = base + lane;
    const bool in = k < cnt && ((S.mask[k] >> warp) & 1u);
    const uint32_t bal = __ballot_sync(0xffffffffu, in);
    if (in) S.list[warp][total + __popc(bal & ((1u << lane) - 1u))] = (uint8_t)k;
    total += __popc(bal);
  }
  if (lane == 0) S.count[warp] = total;
  __syncwarp();
}

// Per-Gaussian, per-column part of p = a2 dx^2 + b2 dx dy + c2 dy^2: f0 = a2 dx^2, g = b2 dx.
struct Col {
  float f0, g;
};
__device__ __forceinline__ Col column(const float4& s0, float dx) {
  return Col{__fmul_rn(__fmul_rn(s0.z, dx), dx), __fmul_rn(s0.w, dx)};
}
// p at row offset dy: dy (c2 dy + g) + f0.  Explicit roundings: the forward and backward
// kernels must evaluate identical bits.
__device__ __forceinline__ float power2(const Col& col, float c2, float dy) {
  return fmaf(dy, fmaf(c2, dy, col.g), col.f0);
}

__device__ __forceinline__ float alpha_of(float opacity, float G) {
  return fminf(kAlphaMax, __fmul_rn(opacity, G));
}

// p passes the skip tests: p_min <= p <= 0 (power <= 0, alpha >= 1/255 before the clamp),
// written as |p - p_min/2| <= -p_min/2 (hm = p_min / 2)
__device__ __forceinline__ bool candidate(float p, float hm) { return fabsf(__fsub_rn(p, hm)) <= -hm; }

// A finished pixel's row coordinate is set to NaN: its power is NaN for every record, and a
// NaN fails the candidate test (every comparison with it is false), so the pixel takes nothing
// more however wide the Gaussian.
__device__ __forceinline__ float parked_row() { return __int_as_float(0x7fc00000); }

template <bool kCount>
__global__ void __launch_bounds__(kThreads, 8) k_render_fwd(const float* __restrict__ proj, int64_t n,
                                                            const uint32_t* __restrict__ vals,
                                                            const uint32_t* __restrict__ ranges, int W, int H,
                                                            int Tx, float3 bg, float* __restrict__ image,
                                                            float* __restrict__ T_final,
                                                            uint32_t* __restrict__ n_contrib,
                                                            uint32_t* __restrict__ work,
                                                            const uint32_t* __restrict__ tile_order,
                                                            uint32_t* __restrict__ tile_cost) {
  __shared__ BatchSmem S;
  __shared__ uint32_t s_cost[kWarps];
  const int tile = tile_order ? (int)__ldg(&tile_order[blockIdx.x]) : (int)blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tile_x0 = (tile % Tx) * gs::kTile, tile_y0 = (tile / Tx) * gs::kTile;
  const int px = tile_x0 + 8 * (warp & 1) + (lane & 7), py0 = tile_y0 + 8 * (warp >> 1) + 2 * (lane >> 3);
  const float fx = (float)px + 0.5f;
  float fy[kPPT];
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  float T[kPPT], cr[kPPT], cg[kPPT], cb[kPPT];
  uint32_t last[kPPT], stop[kPPT], used[kPPT];
  bool done[kPPT];
#pragma unroll
  for (int i = 0; i < kPPT; ++i) {
    fy[i] = (float)(py0 + i) + 0.5f;
    T[i] = 1.f;
    cr[i] = cg[i] = cb[i] = 0.f;
    last[i] = used[i] = 0;
    stop[i] = end - start;  // entries evaluated if the pixel never saturates
    done[i] = !(px < W && py0 + i < H);
  }
#pragma unroll
  for (int i = 0; i < kPPT; ++i)
    if (done[i]) fy[i] = parked_row();
  bool warp_done = __all_sync(0xffffffffu, done[0] && done[1]);
  uint32_t walked = 0;  // entries of this warp's culled lists walked (the same in every lane)
  for (uint32_t b0 = start; b0 < end; b0 += kBatch) {
    if (__syncthreads_count(warp_done) == kThreads) break;
    const int cnt = (int)min((uint32_t)kBatch, end - b0);
#pragma unroll
    for (int r = 0; r < kPerThreadLoad; ++r) {
      const int slot = r * kThreads + threadIdx.x;
      if (slot < cnt) gather_record(proj, n, __ldg(&vals[b0 + slot]), tile_x0, tile_y0, S, slot);
    }
    __syncthreads();
    build_list(S, cnt, warp, lane);
    const int nl = (int)S.count[warp];
    for (int q0 = 0; q0 < nl && !warp_done; q0 += 16) {
      const int qend = min(nl, q0 + 16);
      bool ended = false;
      // two entries per iteration: both candidate tests are independent of the compositing
      // state, so they are issued together; the entries are then composited in list order
      if (kCount) walked += (uint32_t)(qend - q0);
      for (int q = q0; q < qend; q += 2) {
        const bool has1 = q + 1 < qend;
        const int k0 = S.list[warp][q];
        const int k1 = has1 ? S.list[warp][q + 1] : k0;
        const float4 a0 = S.s0[k0], c0 = S.s1[k0];
        const float4 a1 = S.s0[k1], c1 = S.s1[k1];
        const Col cl0 = column(a0, fx - a0.x);
        const Col cl1 = column(a1, fx - a1.x);
        float p0[kPPT], p1[kPPT];
        bool h0[kPPT], h1[kPPT];
#pragma unroll
        for (int i = 0; i < kPPT; ++i) {
          p0[i] = power2(cl0, c0.x, fy[i] - a0.y);
          p1[i] = power2(cl1, c1.x, fy[i] - a1.y);
          h0[i] = candidate(p0[i], c0.z);
          h1[i] = has1 && candidate(p1[i], c1.z);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = e ? k1 : k0;
          const float4 c = e ? c1 : c0;
          bool hit[kPPT];
          float p[kPPT];
#pragma unroll
          for (int i = 0; i < kPPT; ++i) {
            // a pixel that finished before this pair has its row parked and fails the candidate
            // test; one may have finished on entry 0 of the pair
            hit[i] = e ? h1[i] && !done[i] : h0[i];
            p[i] = e ? p1[i] : p0[i];
          }
          if (!__any_sync(0xffffffffu, hit[0] || hit[1])) continue;  // warp-uniform skip
          const float4 col = S.s2[k];
          const uint32_t pos = b0 - start + (uint32_t)k;
          // branch-free per pixel: a pixel that does not take the entry gets weight 0 and
          // keeps its state (fmaf(0, c, x) == x)
#pragma unroll
          for (int i = 0; i < kPPT; ++i) {
            const float alpha = alpha_of(c.y, fast_exp2(p[i]));
            const float Tn = fmaf(-alpha, T[i], T[i]);  // T (1 - alpha), for the stop test
            const bool take = hit[i] && alpha >= kAlphaMin;
            const bool term = take && Tn < kTMin;  // stop before this entry
            const bool acc = take && !term;
            const float w = acc ? alpha * T[i] : 0.f;
            cr[i] = fmaf(w, col.x, cr[i]);
            cg[i] = fmaf(w, col.y, cg[i]);
            cb[i] = fmaf(w, col.z, cb[i]);
            T[i] -= w;  // T (1 - alpha) if taken (within an ulp of Tn), else unchanged
            last[i] = acc ? pos + 1u : last[i];
            if (kCount) used[i] += acc ? 1u : 0u;
            if (term) {  // at most once per pixel: a branch that is almost never taken
              done[i] = true;
              fy[i] = parked_row();
              stop[i] = pos + 1u;
              ended = true;
            }
          }
        }
      }
      if (__any_sync(0xffffffffu, ended)) warp_done = __all_sync(0xffffffffu, done[0] && done[1]);
    }
    __syncthreads();
  }
  if (tile_cost) {  // the backward's walk over this tile: the largest n_contrib of its pixels
    uint32_t lm = 0;
#pragma unroll
    for (int i = 0; i < kPPT; ++i) lm = max(lm, last[i]);
    const uint32_t wmax = __reduce_max_sync(0xffffffffu, lm);
    if (lane == 0) s_cost[warp] = wmax;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t c = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) c = max(c, s_cost[w]);
      tile_cost[tile] = c;
    }
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
      if (kCount) {
        work[pix] = stop[i];
        work[P + pix] = used[i];
        work[2 * P + pix] = walked;
      }
    }
  }
}

// Warp sums of 16 per-lane values by a transposed butterfly: four halving levels (8 + 4 + 2 + 1 shuffles) leave lane L holding
// value (L >> 1) summed over 16 lanes; one plain level finishes it, in lanes 2k and 2k + 1.
__device__ __forceinline__ float warp_transpose_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int level = 0; level < 4; ++level) {
    const int off = 16 >> level;  // 16, 8, 4, 2
    const int half = 8 >> level;  // values kept: 8, 4, 2, 1
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float give = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Two values: one halving level leaves lanes 0..15 with value 0 and 16..31 with value 1,
// four plain levels finish the sums.
__device__ __forceinline__ float warp_transpose_sum2(const float (&v)[2], int lane) {
  const bool upper = (lane & 16) != 0;
  float t = (upper ? v[1] : v[0]) + __shfl_xor_sync(0xffffffffu, upper ? v[0] : v[1], 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 7) k_render_bwd(const float* __restrict__ proj, int64_t n,
                                                            const uint32_t* __restrict__ vals,
                                                            const uint32_t* __restrict__ ranges, int W, int H,
                                                            int Tx, float3 bg, const float* __restrict__ T_final,
                                                            const uint32_t* __restrict__ n_contrib,
                                                            const float* __restrict__ dimg,
                                                            float* __restrict__ grad2d,
                                                            const uint32_t* __restrict__ tile_order) {
  __shared__ BatchSmem S;
  __shared__ uint32_t s_max_last;
  const int tile = tile_order ? (int)__ldg(&tile_order[blockIdx.x]) : (int)blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tile_x0 = (tile % Tx) * gs::kTile, tile_y0 = (tile / Tx) * gs::kTile;
  const int px = tile_x0 + 8 * (warp & 1) + (lane & 7), py0 = tile_y0 + 8 * (warp >> 1) + 2 * (lane >> 3);
  const float fx = (float)px + 0.5f;
  const uint32_t start = ranges[2 * tile], end = ranges[2 * tile + 1];
  const int64_t P = (int64_t)W * H;
  float fy[kPPT], T[kPPT], dr[kPPT], dg[kPPT], db[kPPT], U[kPPT];
  uint32_t last[kPPT];
  uint32_t my_max = 0;
#pragma unroll
  for (int i = 0; i < kPPT; ++i) {
    const int py = py0 + i;
    fy[i] = (float)py + 0.5f;
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
    // U = (colour composited behind the current entry) . dL/dpixel, starting with the
    // background; the colour itself is never needed, only its dot product with dL/dpixel
    U[i] = T[i] * (bg.x * dr[i] + bg.y * dg[i] + bg.z * db[i]);
    my_max = max(my_max, last[i]);
  }
  if (threadIdx.x == 0) s_max_last = 0;
  __syncthreads();
  const uint32_t warp_max = __reduce_max_sync(0xffffffffu, my_max);
  if (lane == 0) atomicMax(&s_max_last, warp_max);
  __syncthreads();
  const uint32_t max_last = s_max_last;
  // batches aligned to the list start, walked from the back
  for (int bb = (int)((max_last + kBatch - 1) / kBatch) - 1; bb >= 0; --bb) {
    const uint32_t b0 = start + (uint32_t)bb * kBatch;
    const int cnt = (int)min((uint32_t)kBatch, min(end, start + max_last) - b0);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kPerThreadLoad; ++r) {
      const int slot = r * kThreads + threadIdx.x;
      if (slot < cnt) gather_record(proj, n, __ldg(&vals[b0 + slot]), tile_x0, tile_y0, S, slot);
    }
    __syncthreads();
    // this warp's list stops at its own pixels' largest n_contrib: no pixel of the warp takes
    // an entry at or past it (the tile's walk runs to the largest over all four warps)
    const uint32_t wend = warp_max > (uint32_t)bb * kBatch ? warp_max - (uint32_t)bb * kBatch : 0u;
    build_list(S, (int)min((uint32_t)cnt, wend), warp, lane);
    const int nl = (int)S.count[warp];
    // two entries per iteration, walked back to front: both candidate tests first (they do
    // not depend on the running state), then the entries in reverse list order
    for (int q = nl - 1; q >= 0; q -= 2) {
      const bool has1 = q >= 1;
      const int k0 = S.list[warp][q];
      const int k1 = has1 ? S.list[warp][q - 1] : k0;
      const uint32_t pos0 = (uint32_t)bb * kBatch + (uint32_t)k0;  // list positions
      const uint32_t pos1 = (uint32_t)bb * kBatch + (uint32_t)k1;
      const float4 a0 = S.s0[k0], c0 = S.s1[k0];
      const float4 a1 = S.s0[k1], c1 = S.s1[k1];
      const Col cl0 = column(a0, fx - a0.x);
      const Col cl1 = column(a1, fx - a1.x);
      float p0[kPPT], p1[kPPT];
      bool h0[kPPT], h1[kPPT];
#pragma unroll
      for (int i = 0; i < kPPT; ++i) {
        p0[i] = power2(cl0, c0.x, fy[i] - a0.y);
        p1[i] = power2(cl1, c1.x, fy[i] - a1.y);
        h0[i] = pos0 < last[i] && candidate(p0[i], c0.z);
        h1[i] = has1 && pos1 < last[i] && candidate(p1[i], c1.z);
      }
      const bool any0 = __any_sync(0xffffffffu, h0[0] || h0[1]);
      const bool any1 = __any_sync(0xffffffffu, h1[0] || h1[1]);
      if (!(any0 || any1)) continue;
      // per entry e: acc[8e + (du, dv, dopacity, dA, dB, dC, dr, dg)] and accb[e] = db
      float acc[16];
      float accb[2] = {0.f, 0.f};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float4 a = e ? a1 : a0;
        const float4 c = e ? c1 : c0;
        bool hit[kPPT];
        float p[kPPT];
#pragma unroll
        for (int i = 0; i < kPPT; ++i) {
          hit[i] = e ? h1[i] : h0[i];
          p[i] = e ? p1[i] : p0[i];
        }
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[8 * e + v] = 0.f;
        if (!(e ? any1 : any0)) continue;  // warp-uniform
        const float4 col = S.s2[e ? k1 : k0];
        const float dx = fx - a.x;
        // moments over the thread's pixels (one column): sum dpow, dpow dy, dpow dy^2.
        // Branch-free per pixel: a pixel that does not take the entry contributes zeros and
        // keeps its state.
        float m0 = 0.f, m1 = 0.f, m2 = 0.f, a6 = 0.f, a7 = 0.f, a2 = 0.f, ab = 0.f;
#pragma unroll
        for (int i = 0; i < kPPT; ++i) {
          const float G = fast_exp2(p[i]);
          const float alpha = alpha_of(c.y, G);
          const bool take = hit[i] && alpha >= kAlphaMin;
          const float dy = fy[i] - a.y;
          const float iom = rcp_approx(__fsub_rn(1.f, alpha));
          T[i] = take ? T[i] * iom : T[i];
          const float w = take ? alpha * T[i] : 0.f;
          a6 = fmaf(w, dr[i], a6);
          a7 = fmaf(w, dg[i], a7);
          ab = fmaf(w, db[i], ab);
          const float cd = col.x * dr[i] + col.y * dg[i] + col.z * db[i];
          const float dalpha = T[i] * cd - U[i] * iom;
          U[i] = fmaf(w, cd, U[i]);
          const bool unclamped = take && __fmul_rn(c.y, G) <= kAlphaMax;
          const float dpow = unclamped ? dalpha * alpha : 0.f;  // d alpha / d power = alpha
          a2 = unclamped ? fmaf(dalpha, G, a2) : a2;
          const float t = dpow * dy;
          m0 += dpow;
          m1 += t;
          m2 = fmaf(t, dy, m2);
        }
        // power = -(A dx^2 + C dy^2)/2 - B dx dy, natural conic from the log2-scaled record
        const float A = a.z * (-2.f / kLog2e), B = a.w * (-1.f / kLog2e), C = c.x * (-2.f / kLog2e);
        const float dxm0 = dx * m0;
        acc[8 * e + 0] = fmaf(A, dxm0, B * m1);
        acc[8 * e + 1] = fmaf(B, dxm0, C * m1);
        acc[8 * e + 2] = a2;
        acc[8 * e + 3] = -0.5f * dx * dxm0;
        acc[8 * e + 4] = -dx * m1;
        acc[8 * e + 5] = -0.5f * m2;
        acc[8 * e + 6] = a6;
        acc[8 * e + 7] = a7;
        accb[e] = ab;
      }
      // both entries' sixteen values in one transposed reduction: lanes 2k, 2k+1 hold value k;
      // the two db values in a second one: lanes 0..15 hold entry 0's, 16..31 entry 1's
      const float tot = warp_transpose_sum16(acc, lane);
      const float tot_b = warp_transpose_sum2(accb, lane);
      if ((lane & 1) == 0) {
        const int kk = lane >> 1, e = kk >> 3, kv = kk & 7;
        if (e ? any1 : any0) {
          float* rec = grad2d + 12 * (int64_t)__float_as_uint(e ? c1.w : c0.w);
          atomicAdd(rec + kv + (kv >= 3 ? 1 : 0) + (kv >= 6 ? 1 : 0), tot);
        }
      } else if (lane == 1 || lane == 17) {
        const int e = lane >> 4;
        if (e ? any1 : any0) atomicAdd(grad2d + 12 * (int64_t)__float_as_uint(e ? c1.w : c0.w) + 10, tot_b);
      }
    }
  }
}

}  // namespace

extern "C" gs_status gs_render_fwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                                   const gs_camera* cam, const float* bg, float* image, float* T_final,
                                   uint32_t* n_contrib, uint32_t* work, const uint32_t* tile_order,
                                   uint32_t* tile_cost, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: bad n");
  if (!ranges || !image || !T_final || !n_contrib || (n > 0 && (!proj || !vals)))
    return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: NULL pointer");
  if (proj && !gs::aligned16(proj)) return gs::set_error(GS_ERR_INVALID, "gs_render_fwd: proj must be 16-byte aligned");
  const gs::Cam k = gs::make_cam(*cam);
  const float3 b = bg ? make_float3(bg[0], bg[1], bg[2]) : make_float3(0.f, 0.f, 0.f);
  cudaStream_t st = gs::as_stream(stream);
  if (work)
    k_render_fwd<true><<<k.Tx * k.Ty, kThreads, 0, st>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, image, T_final,
                                                          n_contrib, work, tile_order, tile_cost);
  else
    k_render_fwd<false><<<k.Tx * k.Ty, kThreads, 0, st>>>(proj, n, vals, ranges, k.W, k.H, k.Tx, b, image, T_final,
                                                           n_contrib, work, tile_order, tile_cost);
  return gs::check_launch("gs_render_fwd");
}

extern "C" gs_status gs_render_bwd(const float* proj, int64_t n, const uint32_t* vals, const uint32_t* ranges,
                                   const gs_camera* cam, const float* bg, const float* T_final,
                                   const uint32_t* n_contrib, const float* dL_dimage, float* grad2d,
                                   const uint32_t* tile_order, void* stream) {
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
                                                 dL_dimage, grad2d, tile_order);
  return gs::check_launch("gs_render_bwd");
}
