// Launch order of the compositing calls' tiles (gs_tile_order): heaviest first.
//
// Tiles carry unequal work and thread blocks start in index order, so a heavy tile issued in
// the last wave runs alone at the end of a launch.  The order ranks the tiles (or square
// blocks of `unit` x `unit` neighbouring tiles, each block's tiles issued together in
// row-major order) by a key of their cost: 0 for a zero cost, else 1 + 16 floor(log2 c) plus
// the four bits of c below its leading one (sixteen steps per octave); a block's key is that
// of its heaviest tile.  A tile's cost is its list length (ranges) or the caller's per-tile
// cost.  One CTA of 1024 threads: a histogram of the keys (weighted by the blocks' tile
// counts), its descending exclusive scan, a scatter by shared-memory atomics (the order of
// blocks with equal keys is unspecified).  Single tiles take a batched path: eight tiles per
// thread per round, all of their loads in flight together.
#include "common.cuh"

namespace {

constexpr int kOrderThreads = 1024;
constexpr int kOrderKeys = 1024;  // keys 0 .. 1 + 16 * 31 + 15
constexpr int kMaxUnit = 8;
constexpr int kBatchTiles = 8;    // single tiles per thread per round
constexpr uint32_t kNoKey = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t cost_key(uint32_t c) {
  if (c == 0u) return 0u;
  const uint32_t hb = 31u - (uint32_t)__clz(c);
  const uint32_t frac = hb >= 4u ? (c >> (hb - 4u)) & 15u : (c << (4u - hb)) & 15u;
  return 1u + 16u * hb + frac;
}

__device__ __forceinline__ uint32_t tile_cost_of(const uint32_t* __restrict__ ranges,
                                                 const uint32_t* __restrict__ cost, int64_t t) {
  return cost ? __ldg(&cost[t]) : __ldg(&ranges[2 * t + 1]) - __ldg(&ranges[2 * t]);
}

// Keys of single tiles t0 + j * kOrderThreads + tid, j < kBatchTiles (kNoKey past T).
__device__ __forceinline__ void tile_keys(const uint32_t* __restrict__ ranges, const uint32_t* __restrict__ cost,
                                          int64_t T, int64_t t0, uint32_t (&key)[kBatchTiles]) {
  uint32_t c[kBatchTiles];
#pragma unroll
  for (int j = 0; j < kBatchTiles; ++j) {
    const int64_t t = t0 + (int64_t)j * kOrderThreads + threadIdx.x;
    c[j] = t < T ? tile_cost_of(ranges, cost, t) : 0u;
  }
#pragma unroll
  for (int j = 0; j < kBatchTiles; ++j) {
    const int64_t t = t0 + (int64_t)j * kOrderThreads + threadIdx.x;
    key[j] = t < T ? cost_key(c[j]) : kNoKey;
  }
}

__global__ void __launch_bounds__(kOrderThreads) k_tile_order(const uint32_t* __restrict__ ranges,
                                                             const uint32_t* __restrict__ cost, int Tx, int Ty,
                                                             int unit, uint32_t* __restrict__ order) {
  __shared__ uint32_t cnt[kOrderKeys];
  __shared__ uint32_t wsum[kOrderThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t T = (int64_t)Tx * Ty;
  const int Ux = (Tx + unit - 1) / unit, Uy = (Ty + unit - 1) / unit;
  const int64_t U = (int64_t)Ux * Uy;
  constexpr int64_t kRound = (int64_t)kOrderThreads * kBatchTiles;
  // block u's key and tile count
  auto block_key = [&](int64_t u, uint32_t& n) {
    const int x0 = (int)(u % Ux) * unit, y0 = (int)(u / Ux) * unit;
    const int w = min(unit, Tx - x0), h = min(unit, Ty - y0);
    n = (uint32_t)(w * h);
    uint32_t m = 0u;
    for (int dy = 0; dy < h; ++dy) {
      const int64_t row = (int64_t)(y0 + dy) * Tx + x0;
#pragma unroll 4
      for (int dx = 0; dx < w; ++dx) m = max(m, tile_cost_of(ranges, cost, row + dx));
    }
    return cost_key(m);
  };
  for (int i = tid; i < kOrderKeys; i += kOrderThreads) cnt[i] = 0u;
  __syncthreads();
  if (unit == 1) {
    for (int64_t t0 = 0; t0 < T; t0 += kRound) {
      uint32_t key[kBatchTiles];
      tile_keys(ranges, cost, T, t0, key);
#pragma unroll
      for (int j = 0; j < kBatchTiles; ++j)
        if (key[j] != kNoKey) atomicAdd(&cnt[key[j]], 1u);
    }
  } else {
    for (int64_t u = tid; u < U; u += kOrderThreads) {
      uint32_t n;
      const uint32_t k = block_key(u, n);
      atomicAdd(&cnt[k], n);
    }
  }
  __syncthreads();
  // thread i takes key kOrderKeys - 1 - i: an exclusive scan in thread order is the
  // descending one
  static_assert(kOrderKeys == kOrderThreads, "one key per thread");
  const int k = kOrderKeys - 1 - tid;
  const uint32_t c = cnt[k];
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  uint32_t woff = 0;
  for (int w = 0; w < warp; ++w) woff += wsum[w];
  cnt[k] = woff + incl - c;
  __syncthreads();
  if (unit == 1) {
    for (int64_t t0 = 0; t0 < T; t0 += kRound) {
      uint32_t key[kBatchTiles];
      tile_keys(ranges, cost, T, t0, key);
#pragma unroll
      for (int j = 0; j < kBatchTiles; ++j)
        if (key[j] != kNoKey) order[atomicAdd(&cnt[key[j]], 1u)] = (uint32_t)(t0 + (int64_t)j * kOrderThreads + tid);
    }
  } else {
    for (int64_t u = tid; u < U; u += kOrderThreads) {
      uint32_t n;
      const uint32_t key = block_key(u, n);
      uint32_t pos = atomicAdd(&cnt[key], n);
      const int x0 = (int)(u % Ux) * unit, y0 = (int)(u / Ux) * unit;
      const int w = min(unit, Tx - x0), h = min(unit, Ty - y0);
      for (int dy = 0; dy < h; ++dy)
        for (int dx = 0; dx < w; ++dx) order[pos++] = (uint32_t)((int64_t)(y0 + dy) * Tx + x0 + dx);
    }
  }
}

}  // namespace

extern "C" gs_status gs_tile_order(const uint32_t* ranges, const uint32_t* tile_cost, int tiles_x, int tiles_y,
                                   int block, uint32_t* order, void* stream) {
  if (tiles_x < 0 || tiles_y < 0 || tiles_x > 65535 || tiles_y > 65535)
    return gs::set_error(GS_ERR_INVALID, "gs_tile_order: tile grid %d x %d out of range", tiles_x, tiles_y);
  if (block < 1 || block > kMaxUnit)
    return gs::set_error(GS_ERR_INVALID, "gs_tile_order: block must be 1..%d", kMaxUnit);
  if (tiles_x == 0 || tiles_y == 0) return GS_OK;
  if (!order || (!tile_cost && !ranges)) return gs::set_error(GS_ERR_INVALID, "gs_tile_order: NULL pointer");
  k_tile_order<<<1, kOrderThreads, 0, gs::as_stream(stream)>>>(ranges, tile_cost, tiles_x, tiles_y, block, order);
  return gs::check_launch("gs_tile_order");
}
