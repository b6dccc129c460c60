// Tile binning and depth sort (gs_bin_sort): duplicate each visible Gaussian into the
// 16x16 tiles of its rectangle with key (tile << 32 | depth bits), then a stable LSD radix
// sort of the (key, index) pairs and per-tile [start, end) ranges.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_scan_dup    single-pass scan of tiles-touched with decoupled look-back; each CTA then
//                 writes its chunk's instances with warp-coalesced stores (the instance
//                 range of a chunk is contiguous, each output slot finds its Gaussian by
//                 binary search in shared memory).  The last chunk publishes M.
//   k_histogram   8-bit digit histograms of every radix pass in one read of the keys;
//                 clears the look-back state of the passes.
//   k_digit_scan  exclusive digit offsets per pass.
//   k_onesweep    one radix pass: persistent CTAs take 4096-key tiles in order from an
//                 atomic counter, rank keys stably in shared memory (warp match-any
//                 ranking), obtain the tile's global digit offsets by decoupled look-back,
//                 and scatter through shared memory so global writes are digit-contiguous.
//   k_ranges      [start, end) of every tile from neighbouring keys.
// Every device-side wait is bounded (gs_debug_set_wait_limit); on expiry the kernel sets
// status bit 2 in count[1] and carries on, so nothing can hang.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanChunk = kScanThreads * kScanItems;  // Gaussians per scan CTA

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;  // keys per radix tile
constexpr int kMaxPasses = 8;

constexpr uint64_t kFlagAgg = 1ull << 62, kFlagPre = 2ull << 62, kValMask = (1ull << 62) - 1;
constexpr uint32_t kFlagAgg32 = 1u << 30, kFlagPre32 = 2u << 30, kValMask32 = (1u << 30) - 1;

struct Workspace {
  uint64_t* keys_alt;
  uint32_t* vals_alt;
  unsigned long long* scan_state;  // per scan chunk
  uint32_t* lookback;               // [pass][tile][256]
  uint32_t* small;                  // counters + histograms, cleared by one memset
  size_t small_bytes;
};
// layout of `small`
constexpr int kSmScanCounter = 0;
constexpr int kSmTileCounters = 1;               // kMaxPasses
constexpr int kSmHist = 16;                      // kMaxPasses * 256
constexpr int kSmDigitBase = 16 + kMaxPasses * 256;
constexpr int kSmWords = 16 + 2 * kMaxPasses * 256;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int tile_bits(int64_t T) {
  int b = 0;
  while ((int64_t(1) << b) < T) ++b;
  return b;
}

int num_passes(const gs::Cam& k) {
  const int tb = tile_bits((int64_t)k.Tx * k.Ty);
  return 4 + (tb + 7) / 8;  // 32 depth bits (sign bit always 0) + tile id bits
}

size_t carve(Workspace* w, char* base, int64_t n, int64_t cap, int passes) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  const int64_t chunks = (n + kScanChunk - 1) / kScanChunk;
  const int64_t tiles = (cap + kSortTile - 1) / kSortTile;
  char* ka = take(sizeof(uint64_t) * (size_t)std::max<int64_t>(cap, 1));
  char* va = take(sizeof(uint32_t) * (size_t)std::max<int64_t>(cap, 1));
  char* ss = take(sizeof(unsigned long long) * (size_t)std::max<int64_t>(chunks, 1));
  char* lb = take(sizeof(uint32_t) * 256 * (size_t)passes * (size_t)std::max<int64_t>(tiles, 1));
  char* sm = take(sizeof(uint32_t) * kSmWords);
  if (w) {
    w->keys_alt = reinterpret_cast<uint64_t*>(ka);
    w->vals_alt = reinterpret_cast<uint32_t*>(va);
    w->scan_state = reinterpret_cast<unsigned long long*>(ss);
    w->lookback = reinterpret_cast<uint32_t*>(lb);
    w->small = reinterpret_cast<uint32_t*>(sm);
    w->small_bytes = sizeof(uint32_t) * kSmWords;
  }
  return off;
}

// Spin on *p until its flag bits are nonzero, at most `limit` iterations.
__device__ __forceinline__ unsigned long long wait_u64(const unsigned long long* p, int64_t limit, bool* timed_out) {
  unsigned long long v = ld_acquire_u64(p);
  for (int64_t it = 0; (v >> 62) == 0; ++it) {
    if (it >= limit) { *timed_out = true; return v; }
    if (it > 32) __nanosleep(64);
    v = ld_acquire_u64(p);
  }
  return v;
}
__device__ __forceinline__ uint32_t wait_u32(const uint32_t* p, int64_t limit, bool* timed_out) {
  uint32_t v = ld_acquire_u32(p);
  for (int64_t it = 0; (v >> 30) == 0; ++it) {
    if (it >= limit) { *timed_out = true; return v; }
    if (it > 32) __nanosleep(64);
    v = ld_acquire_u32(p);
  }
  return v;
}

// ------------------------------------------------------------------ scan + duplicate
__global__ void __launch_bounds__(kScanThreads) k_scan_dup(const float* __restrict__ proj, int64_t n, gs::Cam k,
                                                            uint64_t* __restrict__ keys, uint32_t* __restrict__ vals,
                                                            int64_t cap, unsigned long long* scan_state,
                                                            uint32_t* small, int64_t* count, int64_t limit) {
  __shared__ uint32_t s_items[kScanChunk];   // tiles touched, then local exclusive offsets
  __shared__ uint32_t s_rect[kScanChunk];    // x0 | y0 << 16
  __shared__ uint32_t s_width[kScanChunk];   // rectangle width in tiles
  __shared__ uint32_t s_zbits[kScanChunk];
  __shared__ uint32_t s_warp[kScanThreads / 32];
  __shared__ unsigned long long s_prefix;
  __shared__ uint32_t s_chunk;
  const int tid = threadIdx.x;
  if (tid == 0) s_chunk = atomicAdd(&small[kSmScanCounter], 1u);
  __syncthreads();
  const int64_t chunk = s_chunk;
  const int64_t nchunks = (n + kScanChunk - 1) / kScanChunk;
  const int64_t base = chunk * kScanChunk;
  const float4* q0 = reinterpret_cast<const float4*>(proj);
  const float4* q1 = q0 + n;
  // striped loads (coalesced), per-Gaussian rectangle recomputed from (u, v, radius)
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    const int li = j * kScanThreads + tid;
    const int64_t i = base + li;
    uint32_t cnt = 0, rect = 0, width = 0, zb = 0;
    if (i < n) {
      const int r = __float_as_int(__ldg(&q1[i].w));
      if (r > 0) {
        const float4 a = __ldg(&q0[i]);
        const int fu = (int)floorf(fminf(fmaxf(a.x, -1e9f), 1e9f));
        const int fv = (int)floorf(fminf(fmaxf(a.y, -1e9f), 1e9f));
        const int x0 = min(max((fu - r) >> 4, 0), k.Tx), x1 = min(max(((fu + r) >> 4) + 1, 0), k.Tx);
        const int y0 = min(max((fv - r) >> 4, 0), k.Ty), y1 = min(max(((fv + r) >> 4) + 1, 0), k.Ty);
        if (x0 < x1 && y0 < y1) {
          cnt = (uint32_t)((x1 - x0) * (y1 - y0));
          rect = (uint32_t)x0 | ((uint32_t)y0 << 16);
          width = (uint32_t)(x1 - x0);
          zb = __float_as_uint(a.z);
        }
      }
    }
    s_items[li] = cnt;
    s_rect[li] = rect;
    s_width[li] = width;
    s_zbits[li] = zb;
  }
  __syncthreads();
  // blocked scan: thread t owns items t*8 .. t*8+7
  uint32_t v[kScanItems];
  uint32_t sum = 0;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    v[j] = s_items[tid * kScanItems + j];
    sum += v[j];
  }
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t incl = sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  uint32_t warp_off = 0, total = 0;
  for (int w = 0; w < kScanThreads / 32; ++w) {
    const uint32_t x = s_warp[w];
    if (w < warp) warp_off += x;
    total += x;
  }
  uint32_t run = warp_off + incl - sum;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    s_items[tid * kScanItems + j] = run;  // exclusive local offset
    run += v[j];
  }
  // chunk prefix by decoupled look-back
  if (tid == 0) {
    unsigned long long excl = 0;
    bool to = false;
    if (chunk == 0) {
      st_release_u64(&scan_state[0], kFlagPre | (unsigned long long)total);
    } else {
      st_release_u64(&scan_state[chunk], kFlagAgg | (unsigned long long)total);
      for (int64_t p = chunk - 1; p >= 0; --p) {
        const unsigned long long s = wait_u64(&scan_state[p], limit, &to);
        if (to) break;
        excl += s & kValMask;
        if ((s >> 62) == 2) break;
      }
      st_release_u64(&scan_state[chunk], kFlagPre | (excl + total));
    }
    if (to) atomicOr(reinterpret_cast<unsigned long long*>(&count[1]), (unsigned long long)gs::kStatusTimeout);
    s_prefix = excl;
    if (chunk == nchunks - 1) {
      const int64_t M = (int64_t)(excl + total);
      count[0] = M;
      if (M > cap) atomicOr(reinterpret_cast<unsigned long long*>(&count[1]), (unsigned long long)gs::kStatusCapacity);
    }
  }
  __syncthreads();
  // cooperative, coalesced write of this chunk's instances
  const int64_t out0 = (int64_t)s_prefix;
  const int nvalid = (int)min((int64_t)kScanChunk, n - base);
  for (uint32_t p = tid; p < total; p += kScanThreads) {
    // last item whose exclusive offset <= p
    int lo = 0, hi = nvalid - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_items[mid] <= p) lo = mid; else hi = mid - 1;
    }
    const uint32_t j = p - s_items[lo];
    const uint32_t w = s_width[lo];
    const uint32_t rect = s_rect[lo];
    const uint32_t tx = (rect & 0xffffu) + j % w, ty = (rect >> 16) + j / w;
    const int64_t o = out0 + p;
    if (o < cap) {
      keys[o] = ((uint64_t)(ty * (uint32_t)k.Tx + tx) << 32) | s_zbits[lo];
      vals[o] = (uint32_t)(base + lo);
    }
  }
}

// ------------------------------------------------------------------ digit histograms
__global__ void __launch_bounds__(256) k_histogram(const uint64_t* __restrict__ keys, int64_t cap, int passes,
                                                    uint32_t* small, uint32_t* lookback, const int64_t* count) {
  __shared__ uint32_t s_hist[kMaxPasses][256];
  if (count[1] != 0) return;
  const int64_t M = min(count[0], cap);
  const int64_t tiles = (M + kSortTile - 1) / kSortTile;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // clear the look-back state of every pass for the tiles in use
  for (int64_t w = gtid; w < (int64_t)passes * tiles * 256; w += stride) {
    const int64_t pass = w / (tiles * 256), rest = w % (tiles * 256);
    lookback[pass * ((cap + kSortTile - 1) / kSortTile) * 256 + rest] = 0u;
  }
  for (int i = threadIdx.x; i < kMaxPasses * 256; i += blockDim.x) (&s_hist[0][0])[i] = 0u;
  __syncthreads();
  for (int64_t i = gtid; i < M; i += stride) {
    const uint64_t key = keys[i];
    for (int p = 0; p < passes; ++p) atomicAdd(&s_hist[p][(key >> (8 * p)) & 255u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < passes * 256; i += blockDim.x) {
    const uint32_t c = (&s_hist[0][0])[i];
    if (c) atomicAdd(&small[kSmHist + i], c);
  }
}

__global__ void k_digit_scan(uint32_t* small, int passes, const int64_t* count) {
  __shared__ uint32_t s[256];
  if (count[1] != 0) return;
  const int t = threadIdx.x;
  for (int p = 0; p < passes; ++p) {
    s[t] = small[kSmHist + p * 256 + t];
    __syncthreads();
    if (t == 0) {
      uint32_t run = 0;
      for (int d = 0; d < 256; ++d) {
        const uint32_t c = s[d];
        s[d] = run;
        run += c;
      }
    }
    __syncthreads();
    small[kSmDigitBase + p * 256 + t] = s[t];
    __syncthreads();
  }
}

// ------------------------------------------------------------------ one radix pass
struct SortSmem {
  uint64_t keys[kSortTile];
  uint32_t vals[kSortTile];
  uint32_t whist[kSortWarps][256];
  uint32_t tstart[256];
  uint32_t gbase[256];
  uint32_t wsum[kSortWarps];
  uint32_t tile;
};

__global__ void __launch_bounds__(kSortThreads) k_onesweep(const uint64_t* __restrict__ kin,
                                                            const uint32_t* __restrict__ vin,
                                                            uint64_t* __restrict__ kout, uint32_t* __restrict__ vout,
                                                            int64_t cap, int pass, uint32_t* small,
                                                            uint32_t* lookback_pass, int64_t* count, int64_t limit,
                                                            int drop_publish) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmem& S = *reinterpret_cast<SortSmem*>(smem_raw);
  if (count[1] != 0) return;
  const int64_t M = min(count[0], cap);
  const int64_t ntiles = (M + kSortTile - 1) / kSortTile;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int shift = 8 * pass;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t* digit_base = small + kSmDigitBase + pass * 256;
  while (true) {
    if (tid == 0) S.tile = atomicAdd(&small[kSmTileCounters + pass], 1u);
    for (int i = tid; i < kSortWarps * 256; i += kSortThreads) (&S.whist[0][0])[i] = 0u;
    __syncthreads();
    const int64_t tile = S.tile;
    if (tile >= ntiles) break;
    const int64_t base = tile * kSortTile;
    const int nvalid = (int)min((int64_t)kSortTile, M - base);
    // ---- load (warp-striped) and rank stably within the warp
    uint64_t k[kSortItems];
    uint32_t v[kSortItems], rank[kSortItems];
    const int wbase = warp * (kSortItems * 32);
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int li = wbase + i * 32 + lane;
      if (li < nvalid) {
        k[i] = kin[base + li];
        v[i] = vin[base + li];
      } else {
        k[i] = ~0ull;
        v[i] = 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int li = wbase + i * 32 + lane;
      const bool valid = li < nvalid;
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t d = (uint32_t)(k[i] >> shift) & 255u;
        const uint32_t peers = __match_any_sync(vmask, d);
        const uint32_t before = S.whist[warp][d];
        __syncwarp(vmask);
        const int leader = 31 - __clz(peers);
        if (lane == leader) S.whist[warp][d] = before + __popc(peers);
        __syncwarp(vmask);
        rank[i] = before + __popc(peers & lt_mask);
      }
    }
    __syncthreads();
    // ---- per digit: prefix over warps, tile count, look-back for the global offset
    {
      const int d = tid;  // 256 threads = 256 digits
      uint32_t run = 0;
#pragma unroll
      for (int w = 0; w < kSortWarps; ++w) {
        const uint32_t c = S.whist[w][d];
        S.whist[w][d] = run;
        run += c;
      }
      const uint32_t cnt = run;
      uint32_t* my = lookback_pass + tile * 256 + d;
      uint32_t excl = 0;
      bool to = false;
      const bool drop = drop_publish && tile == 0;
      if (tile == 0) {
        if (!drop) st_release_u32(my, kFlagPre32 | cnt);
      } else {
        st_release_u32(my, kFlagAgg32 | cnt);
        for (int64_t p = tile - 1; p >= 0; --p) {
          const uint32_t s = wait_u32(lookback_pass + p * 256 + d, limit, &to);
          if (to) break;
          excl += s & kValMask32;
          if ((s >> 30) == 2) break;
        }
        st_release_u32(my, kFlagPre32 | ((excl + cnt) & kValMask32));
      }
      if (to) atomicOr(reinterpret_cast<unsigned long long*>(&count[1]), (unsigned long long)gs::kStatusTimeout);
      S.gbase[d] = digit_base[d] + excl;
      // exclusive scan of the tile's digit counts
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) S.wsum[warp] = incl;
      __syncthreads();
      uint32_t woff = 0;
      for (int w = 0; w < warp; ++w) woff += S.wsum[w];
      S.tstart[d] = woff + incl - cnt;
    }
    __syncthreads();
    // ---- scatter into shared memory in tile order
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int li = wbase + i * 32 + lane;
      if (li < nvalid) {
        const uint32_t d = (uint32_t)(k[i] >> shift) & 255u;
        const uint32_t pos = S.tstart[d] + S.whist[warp][d] + rank[i];
        S.keys[pos] = k[i];
        S.vals[pos] = v[i];
      }
    }
    __syncthreads();
    // ---- digit-contiguous global writes
#pragma unroll 4
    for (int i = 0; i < kSortItems; ++i) {
      const int p = i * kSortThreads + tid;
      if (p < nvalid) {
        const uint64_t key = S.keys[p];
        const uint32_t d = (uint32_t)(key >> shift) & 255u;
        const uint32_t g = S.gbase[d] + (uint32_t)p - S.tstart[d];
        if (g < (uint64_t)M) {  // always true unless a look-back wait gave up (status bit set)
          kout[g] = key;
          vout[g] = S.vals[p];
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ tile ranges
__global__ void k_ranges(const uint64_t* __restrict__ keys, int64_t cap, uint32_t* __restrict__ ranges,
                         const int64_t* count) {
  if (count[1] != 0) return;
  const int64_t M = min(count[0], cap);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < M; i += stride) {
    const uint32_t t = (uint32_t)(keys[i] >> 32);
    if (i == 0 || (uint32_t)(keys[i - 1] >> 32) != t) ranges[2 * (int64_t)t] = (uint32_t)i;
    if (i == M - 1 || (uint32_t)(keys[i + 1] >> 32) != t) ranges[2 * (int64_t)t + 1] = (uint32_t)(i + 1);
  }
}

int sort_blocks_per_sm() {
  static int cached = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (cached < 0) {
    int b = 0;
    cudaFuncSetAttribute(k_onesweep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SortSmem));
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_onesweep, kSortThreads, sizeof(SortSmem)) != cudaSuccess ||
        b < 1)
      b = 1;
    cached = b;
  }
  return cached;
}

}  // namespace

extern "C" size_t gs_bin_sort_workspace_size(int64_t n, int64_t capacity, const gs_camera* cam) {
  if (!cam || n < 0 || capacity < 0) return 0;
  const gs::Cam k = gs::make_cam(*cam);
  return carve(nullptr, nullptr, n, capacity, num_passes(k));
}

extern "C" gs_status gs_bin_sort(const float* proj, int64_t n, const gs_camera* cam, void* workspace,
                                 size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                                 uint32_t* ranges, int64_t* count, int64_t* count_host, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n > (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: bad n");
  if (capacity < 0 || capacity >= (int64_t(1) << 30))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: capacity must be in [0, 2^30)");
  if (!count || !ranges || (n > 0 && !proj) || (capacity > 0 && (!keys || !vals)) || !workspace)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: NULL pointer");
  if ((proj && !gs::aligned16(proj)) || !gs::aligned8(count) || (keys && !gs::aligned8(keys)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: misaligned pointer");
  const gs::Cam k = gs::make_cam(*cam);
  const int passes = num_passes(k);
  if (passes > kMaxPasses) return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: too many tiles");
  const size_t need = carve(nullptr, nullptr, n, capacity, passes);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: workspace %zu bytes < %zu needed", workspace_bytes, need);
  Workspace w;
  carve(&w, reinterpret_cast<char*>(workspace), n, capacity, passes);
  cudaStream_t st = gs::as_stream(stream);
  const int64_t T = (int64_t)k.Tx * k.Ty;
  const int64_t limit = gs::wait_limit();
  const int drop = gs::take_drop_publish();

  if (cudaMemsetAsync(count, 0, 2 * sizeof(int64_t), st) != cudaSuccess ||
      cudaMemsetAsync(w.small, 0, w.small_bytes, st) != cudaSuccess ||
      cudaMemsetAsync(ranges, 0, sizeof(uint32_t) * 2 * T, st) != cudaSuccess)
    return gs::check_launch("gs_bin_sort memset");
  if (n > 0) {
    const int64_t chunks = (n + kScanChunk - 1) / kScanChunk;
    if (cudaMemsetAsync(w.scan_state, 0, sizeof(unsigned long long) * chunks, st) != cudaSuccess)
      return gs::check_launch("gs_bin_sort memset");
    // ping-pong so that the last pass lands in the caller's arrays
    uint64_t* ka = (passes % 2 == 0) ? keys : w.keys_alt;
    uint32_t* va = (passes % 2 == 0) ? vals : w.vals_alt;
    uint64_t* kb = (passes % 2 == 0) ? w.keys_alt : keys;
    uint32_t* vb = (passes % 2 == 0) ? w.vals_alt : vals;
    k_scan_dup<<<(unsigned)chunks, kScanThreads, 0, st>>>(proj, n, k, ka, va, capacity, w.scan_state, w.small, count,
                                                           limit);
    if (gs_status s = gs::check_launch("gs_bin_sort scan")) return s;
    const int sms = gs::num_sms();
    k_histogram<<<sms * 4, 256, 0, st>>>(ka, capacity, passes, w.small, w.lookback, count);
    k_digit_scan<<<1, 256, 0, st>>>(w.small, passes, count);
    if (gs_status s = gs::check_launch("gs_bin_sort histogram")) return s;
    const int grid = sms * sort_blocks_per_sm();
    const int64_t max_tiles = (capacity + kSortTile - 1) / kSortTile;
    for (int p = 0; p < passes; ++p) {
      k_onesweep<<<grid, kSortThreads, sizeof(SortSmem), st>>>(ka, va, kb, vb, capacity, p, w.small,
                                                                w.lookback + (size_t)p * max_tiles * 256, count,
                                                                limit, p == 0 ? drop : 0);
      std::swap(ka, kb);
      std::swap(va, vb);
    }
    if (gs_status s = gs::check_launch("gs_bin_sort onesweep")) return s;
    k_ranges<<<sms * 4, 256, 0, st>>>(keys, capacity, ranges, count);
    if (gs_status s = gs::check_launch("gs_bin_sort ranges")) return s;
  }
  if (count_host) {
    int64_t hc[2] = {0, 0};
    if (cudaMemcpyAsync(hc, count, sizeof(hc), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return gs::check_launch("gs_bin_sort count readback");
    *count_host = hc[0];
    if (hc[1] & gs::kStatusTimeout) return gs::set_error(GS_ERR_TIMEOUT, "gs_bin_sort: a look-back wait gave up");
    if (hc[1] & gs::kStatusCapacity)
      return gs::set_error(GS_ERR_CAPACITY, "gs_bin_sort: %lld instances exceed capacity %lld", (long long)hc[0],
                           (long long)capacity);
  }
  return GS_OK;
}
