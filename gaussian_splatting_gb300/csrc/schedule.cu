// Scheduling helpers over the step's own outputs (gs_tile_split, gs_view_order).
//
// gs_tile_split: the pixel-wise load balancing of the Grendel-GS notes (§3.1): the cost of
// every 16x16 pixel block, its cumulative sum, and the split points that give each of K
// parts about Total / K.  Costs are integers (per-pixel work counts of the compositing
// forward), so the sums and split points are exact.  Split k = the number of blocks whose
// inclusive cumulative cost is at most k Total / K (searchsorted on the right), compared as
// K C[i] <= k Total in 128-bit integers.
//   k_tile_cost   one CTA per block: its 256 pixels' costs summed in 64 bits.
//   k_tile_scan   one CTA: the inclusive scan of the block costs, then one binary search per
//                 split point on the (non-decreasing) cumulative sum.
//
// gs_view_order: the Odin summary's scheduling score s(v | U_prev) = sum of the Jaccard
// weights w_uv over the previous set, on the B x B weights gs_visible_sets computes.  Views
// are taken one at a time into task units of `unit` views; the next is the unscheduled view
// with the smallest score against the previous unit (ties: the lower index).
//   k_view_order  one CTA of 64 threads: a thread per candidate view sums its weights over
//                 the previous unit in scheduling order (float32), thread 0 picks the least.
#include "common.cuh"

namespace {

constexpr int kScanThreads = 1024;
constexpr int kMaxParts = 1024;
constexpr int kMaxOrderViews = 64;

__global__ void __launch_bounds__(256) k_tile_cost(const uint32_t* __restrict__ cost, int W, int H, int Tx,
                                                   uint64_t* __restrict__ tile_cost) {
  __shared__ unsigned long long s_part[8];
  const int t = blockIdx.x;
  const int tx = t % Tx, ty = t / Tx;
  const int x = tx * 16 + (threadIdx.x & 15), y = ty * 16 + (threadIdx.x >> 4);
  unsigned long long v = (x < W && y < H) ? (unsigned long long)cost[(int64_t)y * W + x] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long s = 0;
    for (int w = 0; w < 8; ++w) s += s_part[w];
    tile_cost[t] = s;
  }
}

__global__ void __launch_bounds__(kScanThreads) k_tile_scan(const uint64_t* __restrict__ tile_cost, int64_t T,
                                                            int K, uint64_t* __restrict__ cum,
                                                            int64_t* __restrict__ bounds) {
  __shared__ unsigned long long s_warp[kScanThreads / 32];
  __shared__ unsigned long long s_total;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (T + kScanThreads - 1) / kScanThreads;
  const int64_t i0 = min(T, (int64_t)tid * per), i1 = min(T, i0 + per);
  unsigned long long sum = 0;
  for (int64_t i = i0; i < i1; ++i) sum += tile_cost[i];
  // exclusive prefix of the chunk sums over the block
  unsigned long long incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    unsigned long long run = 0;
    for (int w = 0; w < kScanThreads / 32; ++w) {
      const unsigned long long c = s_warp[w];
      s_warp[w] = run;
      run += c;
    }
    s_total = run;
  }
  __syncthreads();
  unsigned long long run = s_warp[warp] + incl - sum;
  for (int64_t i = i0; i < i1; ++i) {
    run += tile_cost[i];
    cum[i] = run;
  }
  __syncthreads();  // cum[] complete and visible to the block
  const unsigned long long total = s_total;
  for (int k = tid; k <= K; k += kScanThreads) {
    int64_t b;
    if (k == 0) {
      b = 0;
    } else if (k == K) {
      b = T;
    } else {  // number of i with K cum[i] <= k total: cum is non-decreasing, so a binary search
      const unsigned __int128 target = (unsigned __int128)k * total;
      int64_t lo = 0, hi = T;  // answer in [lo, hi]
      while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if ((unsigned __int128)K * cum[mid] <= target) lo = mid + 1;
        else hi = mid;
      }
      b = lo;
    }
    bounds[k] = b;
  }
}

__global__ void __launch_bounds__(kMaxOrderViews) k_view_order(const float* __restrict__ w, int B, int unit,
                                                               int32_t* __restrict__ order, float* __restrict__ score) {
  __shared__ float s_w[kMaxOrderViews * kMaxOrderViews];
  __shared__ float s_s[kMaxOrderViews];
  __shared__ int s_prev[kMaxOrderViews], s_cur[kMaxOrderViews];
  __shared__ int s_nprev, s_ncur;
  __shared__ unsigned long long s_done;
  const int v = threadIdx.x;
  for (int i = v; i < B * B; i += kMaxOrderViews) s_w[i] = w[i];
  if (v == 0) {
    s_nprev = 0;
    s_ncur = 0;
    s_done = 0ull;
  }
  __syncthreads();
  for (int k = 0; k < B; ++k) {
    if (v < B) {  // this candidate's score against the previous unit, in its scheduling order
      float s = 0.f;
      for (int j = 0; j < s_nprev; ++j) s += s_w[s_prev[j] * B + v];
      s_s[v] = s;
    }
    __syncthreads();
    if (v == 0) {
      int best = -1;
      float best_s = 0.f;
      for (int c = 0; c < B; ++c) {
        if ((s_done >> c) & 1ull) continue;
        if (best < 0 || s_s[c] < best_s) {
          best = c;
          best_s = s_s[c];
        }
      }
      s_done |= 1ull << best;
      order[k] = best;
      score[k] = best_s;
      s_cur[s_ncur++] = best;
      if (s_ncur == unit) {
        for (int j = 0; j < unit; ++j) s_prev[j] = s_cur[j];
        s_nprev = unit;
        s_ncur = 0;
      }
    }
    __syncthreads();
  }
}

}  // namespace

extern "C" gs_status gs_tile_split(const uint32_t* cost_px, int width, int height, int parts, uint64_t* tile_cost,
                                   uint64_t* cum, int64_t* bounds, void* stream) {
  if (width <= 0 || height <= 0 || width > 32768 || height > 32768)
    return gs::set_error(GS_ERR_INVALID, "gs_tile_split: bad image size %d x %d", width, height);
  if (parts < 1 || parts > kMaxParts)
    return gs::set_error(GS_ERR_INVALID, "gs_tile_split: parts must be 1..%d", kMaxParts);
  if (!cost_px || !tile_cost || !cum || !bounds) return gs::set_error(GS_ERR_INVALID, "gs_tile_split: NULL pointer");
  if (!gs::aligned8(tile_cost) || !gs::aligned8(cum) || !gs::aligned8(bounds))
    return gs::set_error(GS_ERR_INVALID, "gs_tile_split: 64-bit arrays must be 8-byte aligned");
  const int Tx = (width + 15) / 16, Ty = (height + 15) / 16;
  const int64_t T = (int64_t)Tx * Ty;
  cudaStream_t st = gs::as_stream(stream);
  k_tile_cost<<<(unsigned)T, 256, 0, st>>>(cost_px, width, height, Tx, tile_cost);
  if (gs_status s = gs::check_launch("gs_tile_split costs")) return s;
  k_tile_scan<<<1, kScanThreads, 0, st>>>(tile_cost, T, parts, cum, bounds);
  return gs::check_launch("gs_tile_split scan");
}

extern "C" gs_status gs_view_order(const float* weights, int batch, int unit, int32_t* order, float* score,
                                   void* stream) {
  if (batch < 1 || batch > kMaxOrderViews)
    return gs::set_error(GS_ERR_INVALID, "gs_view_order: batch must be 1..%d", kMaxOrderViews);
  if (unit < 1 || unit > batch) return gs::set_error(GS_ERR_INVALID, "gs_view_order: unit must be 1..batch");
  if (!weights || !order || !score) return gs::set_error(GS_ERR_INVALID, "gs_view_order: NULL pointer");
  k_view_order<<<1, kMaxOrderViews, 0, gs::as_stream(stream)>>>(weights, batch, unit, order, score);
  return gs::check_launch("gs_view_order");
}
