// Tile binning and depth sort (gs_bin_sort).
//
// Result (the contract): every visible Gaussian duplicated once per tile of its rectangle
// with key (tile << 32 | float bits of depth) and value = Gaussian index, ordered by
// (tile, depth, index), plus per-tile [start, end) ranges.
//
// How: a stable sort by tile of a list that is already in (depth, index) order is the sort
// by (tile, depth, index).  So the N Gaussians are sorted once by depth (4 stable radix
// passes over 32-bit keys; equal depths keep index order), the instances are emitted in
// that order as (tile, index) pairs, and only the tile ids of the M instances are
// radix-sorted (ceil(log2(tiles) / 8) passes: 2 for up to 65,536 tiles) on 8-byte pairs --
// about a third of the traffic of sorting all 64 key bits of 12-byte pairs.
//
// Kernels (all on the caller's stream, no host synchronisation):
//   k_depth_init  depth keys (0xFFFFFFFF for culled Gaussians) + their digit histograms;
//                 clears the look-back state of every pass.
//   k_digit_scan  exclusive digit offsets per pass.
//   k_onesweep    one stable radix pass of 8 bits: persistent CTAs take 4096-key tiles in
//                 order from an atomic counter, rank keys within the tile in shared memory
//                 (warp match-any ranking), get the tile's global digit offsets by
//                 decoupled look-back and scatter through shared memory so the global
//                 writes are digit-contiguous.
//   k_scan_dup    single-pass scan (decoupled look-back) of tiles-touched over the depth-
//                 sorted Gaussians; each CTA writes its contiguous run of (tile, index)
//                 pairs with coalesced stores and adds the run's tile-digit histograms.
//                 The last chunk publishes M.
//   k_finalize    64-bit keys (tile << 32 | depth bits), values, and every tile's
//                 [start, end) from neighbouring tile ids.
// Every device-side wait is bounded (gs_debug_set_wait_limit); on expiry the kernel sets
// status bit 2 in count[1] and carries on, so nothing can hang.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanItems = 2;
constexpr int kScanChunk = kScanThreads * kScanItems;  // Gaussians per scan CTA
constexpr int kWin = 4096;                             // output slots per write window
constexpr int kWinPer = kWin / kScanThreads;

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kDepthItems = 4;    // depth passes: 1024 keys per radix tile (N is modest)
constexpr int kTileItems = 12;    // tile passes: 3072 keys per radix tile (M is large)
constexpr int kDepthPasses = 4;
constexpr int kMaxTilePasses = 4;
constexpr int kSlots = kDepthPasses + kMaxTilePasses;  // histogram / counter slots

constexpr uint64_t kFlagAgg = 1ull << 62, kFlagPre = 2ull << 62, kValMask = (1ull << 62) - 1;
constexpr uint32_t kFlagAgg32 = 1u << 30, kFlagPre32 = 2u << 30, kValMask32 = (1u << 30) - 1;
constexpr uint32_t kCulledKey = 0xFFFFFFFFu;

// layout of the small, memset-cleared block of the workspace (32-bit words)
constexpr int kSmScanCounter = 0;
constexpr int kSmTileCounters = 1;  // kSlots
constexpr int kSmHist = 16;         // kSlots * 256
constexpr int kSmDigitBase = kSmHist + kSlots * 256;
constexpr int kSmWords = kSmDigitBase + kSlots * 256;

struct Workspace {
  uint32_t* tkey[2];               // instance tile ids, ping-pong
  uint32_t* tval[2];               // instance Gaussian indices, ping-pong
  uint32_t* dkey[2];
  uint32_t* didx[2];
  unsigned long long* scan_state;  // per scan chunk
  uint32_t* lb_depth;              // [pass][tile][256]
  uint32_t* lb_tile;               // [pass][tile][256]
  uint32_t* small;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
template <int ITEMS>
__host__ __device__ inline int64_t sort_tiles(int64_t m) {
  constexpr int kTile = kSortThreads * ITEMS;
  return (m + kTile - 1) / kTile;
}

int tile_bits(int64_t T) {
  int b = 0;
  while ((int64_t(1) << b) < T) ++b;
  return b;
}

int tile_passes(const gs::Cam& k) { return std::max(1, (tile_bits((int64_t)k.Tx * k.Ty) + 7) / 8); }

size_t carve(Workspace* w, char* base, int64_t n, int64_t cap, int tpasses) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align256(std::max<size_t>(bytes, 1));
    return p;
  };
  const int64_t chunks = (n + kScanChunk - 1) / kScanChunk;
  char* tk0 = take(sizeof(uint32_t) * (size_t)cap);
  char* tk1 = take(sizeof(uint32_t) * (size_t)cap);
  char* tv0 = take(sizeof(uint32_t) * (size_t)cap);
  char* tv1 = take(sizeof(uint32_t) * (size_t)cap);
  char* dk0 = take(sizeof(uint32_t) * (size_t)n);
  char* dk1 = take(sizeof(uint32_t) * (size_t)n);
  char* di0 = take(sizeof(uint32_t) * (size_t)n);
  char* di1 = take(sizeof(uint32_t) * (size_t)n);
  char* ss = take(sizeof(unsigned long long) * (size_t)chunks);
  char* lbd = take(sizeof(uint32_t) * 256 * kDepthPasses * (size_t)sort_tiles<kDepthItems>(n));
  char* lbt = take(sizeof(uint32_t) * 256 * (size_t)tpasses * (size_t)sort_tiles<kTileItems>(cap));
  char* sm = take(sizeof(uint32_t) * kSmWords);
  if (w) {
    w->tkey[0] = reinterpret_cast<uint32_t*>(tk0);
    w->tkey[1] = reinterpret_cast<uint32_t*>(tk1);
    w->tval[0] = reinterpret_cast<uint32_t*>(tv0);
    w->tval[1] = reinterpret_cast<uint32_t*>(tv1);
    w->dkey[0] = reinterpret_cast<uint32_t*>(dk0);
    w->dkey[1] = reinterpret_cast<uint32_t*>(dk1);
    w->didx[0] = reinterpret_cast<uint32_t*>(di0);
    w->didx[1] = reinterpret_cast<uint32_t*>(di1);
    w->scan_state = reinterpret_cast<unsigned long long*>(ss);
    w->lb_depth = reinterpret_cast<uint32_t*>(lbd);
    w->lb_tile = reinterpret_cast<uint32_t*>(lbt);
    w->small = reinterpret_cast<uint32_t*>(sm);
  }
  return off;
}

__device__ __forceinline__ void flag_status(int64_t* count, int64_t bits) {
  atomicOr(reinterpret_cast<unsigned long long*>(&count[1]), (unsigned long long)bits);
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

// ------------------------------------------------------------------ depth keys
__global__ void __launch_bounds__(256) k_depth_init(const float* __restrict__ proj, int64_t n,
                                                     uint32_t* __restrict__ dkey, uint32_t* __restrict__ didx,
                                                     uint32_t* small, uint32_t* lb_depth, uint32_t* lb_tile,
                                                     int64_t lb_tile_words) {
  __shared__ uint32_t s_hist[kDepthPasses][256];
  const float4* q0 = reinterpret_cast<const float4*>(proj);
  const float4* q1 = q0 + n;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t w = gtid; w < (int64_t)kDepthPasses * sort_tiles<kDepthItems>(n) * 256; w += stride) lb_depth[w] = 0u;
  for (int64_t w = gtid; w < lb_tile_words; w += stride) lb_tile[w] = 0u;
  for (int i = threadIdx.x; i < kDepthPasses * 256; i += blockDim.x) (&s_hist[0][0])[i] = 0u;
  __syncthreads();
  for (int64_t i = gtid; i < n; i += stride) {
    const int r = __float_as_int(__ldg(&q1[i].w));
    const uint32_t key = r > 0 ? __float_as_uint(__ldg(&q0[i].z)) : kCulledKey;
    dkey[i] = key;
    didx[i] = (uint32_t)i;
#pragma unroll
    for (int p = 0; p < kDepthPasses; ++p) atomicAdd(&s_hist[p][(key >> (8 * p)) & 255u], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kDepthPasses * 256; i += blockDim.x) {
    const uint32_t c = (&s_hist[0][0])[i];
    if (c) atomicAdd(&small[kSmHist + i], c);
  }
}

// exclusive digit offsets of slots [slot0, slot0 + nslots)
__global__ void k_digit_scan(uint32_t* small, int slot0, int nslots, const int64_t* count) {
  __shared__ uint32_t s_warp[8];
  if (count[1] != 0) return;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int p = slot0; p < slot0 + nslots; ++p) {
    const uint32_t c = small[kSmHist + p * 256 + t];
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t woff = 0;
    for (int w = 0; w < warp; ++w) woff += s_warp[w];
    small[kSmDigitBase + p * 256 + t] = woff + incl - c;
    __syncthreads();
  }
}

// ------------------------------------------------------------------ one stable radix pass
template <int ITEMS>
struct SortSmem {
  uint32_t keys[kSortThreads * ITEMS];
  uint32_t vals[kSortThreads * ITEMS];
  uint32_t whist[kSortWarps][256];
  uint32_t tstart[256];
  uint32_t gbase[256];
  uint32_t wsum[kSortWarps];
  uint32_t tile;
};

// Stable pass over 32-bit keys (8-bit digit at `shift`).  n_host >= 0: sort n_host keys;
// otherwise min(count[0], cap) keys.
template <int ITEMS>
__global__ void __launch_bounds__(kSortThreads, 4) k_onesweep(const uint32_t* __restrict__ kin,
                                                               const uint32_t* __restrict__ vin,
                                                               uint32_t* __restrict__ kout, uint32_t* __restrict__ vout,
                                                               int64_t n_host, int64_t cap, int shift, int slot,
                                                               uint32_t* small, uint32_t* lookback_pass,
                                                               int64_t* count, int64_t limit, int drop_publish) {
  constexpr int kTile = kSortThreads * ITEMS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmem<ITEMS>& S = *reinterpret_cast<SortSmem<ITEMS>*>(smem_raw);
  if (count[1] != 0) return;
  const int64_t M = n_host >= 0 ? n_host : min(count[0], cap);
  const int64_t ntiles = sort_tiles<ITEMS>(M);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const uint32_t* digit_base = small + kSmDigitBase + slot * 256;
  while (true) {
    if (tid == 0) S.tile = atomicAdd(&small[kSmTileCounters + slot], 1u);
    for (int i = tid; i < kSortWarps * 256; i += kSortThreads) (&S.whist[0][0])[i] = 0u;
    __syncthreads();
    const int64_t tile = S.tile;
    if (tile >= ntiles) break;
    const int64_t base = tile * kTile;
    const int nvalid = (int)min((int64_t)kTile, M - base);
    const bool full = nvalid == kTile;
    // ---- load (warp-striped) and rank stably within the warp
    uint32_t k[ITEMS], v[ITEMS], rank[ITEMS];
    const int wbase = warp * (ITEMS * 32);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int li = wbase + i * 32 + lane;
      if (full || li < nvalid) {
        k[i] = kin[base + li];
        v[i] = vin[base + li];
      } else {
        k[i] = 0xFFFFFFFFu;
        v[i] = 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int li = wbase + i * 32 + lane;
      const bool valid = full || li < nvalid;
      const uint32_t vmask = full ? 0xffffffffu : __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t d = (k[i] >> shift) & 255u;
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
      if (tile == 0) {
        if (!drop_publish) st_release_u32(my, kFlagPre32 | cnt);
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
      if (to) flag_status(count, gs::kStatusTimeout);
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
    for (int i = 0; i < ITEMS; ++i) {
      const int li = wbase + i * 32 + lane;
      if (full || li < nvalid) {
        const uint32_t d = (k[i] >> shift) & 255u;
        const uint32_t pos = S.tstart[d] + S.whist[warp][d] + rank[i];
        S.keys[pos] = k[i];
        S.vals[pos] = v[i];
      }
    }
    __syncthreads();
    // ---- digit-contiguous global writes
#pragma unroll 4
    for (int i = 0; i < ITEMS; ++i) {
      const int p = i * kSortThreads + tid;
      if (p < nvalid) {
        const uint32_t key = S.keys[p];
        const uint32_t d = (key >> shift) & 255u;
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

// ------------------------------------------------------------------ scan + duplicate
// Walks the Gaussians in depth order (skey / sidx: depth-sorted keys and indices) and writes
// (tile id, Gaussian index) pairs; also accumulates the tile-digit histograms of the pairs.
__global__ void __launch_bounds__(kScanThreads) k_scan_dup(const float* __restrict__ proj, int64_t n,
                                                            const uint32_t* __restrict__ skey,
                                                            const uint32_t* __restrict__ sidx, gs::Cam k, int tpasses,
                                                            uint32_t* __restrict__ tkey, uint32_t* __restrict__ tval,
                                                            int64_t cap, unsigned long long* scan_state,
                                                            uint32_t* small, int64_t* count, int64_t limit) {
  __shared__ uint32_t s_items[kScanChunk];   // tiles touched, then local exclusive offsets
  __shared__ uint32_t s_rect[kScanChunk];    // x0 | y0 << 16
  __shared__ uint32_t s_width[kScanChunk];   // rectangle width in tiles
  __shared__ uint32_t s_gauss[kScanChunk];
  __shared__ float s_rcpw[kScanChunk];        // 1 / width
  __shared__ uint32_t s_owner[kWin];          // owner of each output slot in the window
  __shared__ uint32_t s_hist[kMaxTilePasses][256];
  __shared__ uint32_t s_warp[kScanThreads / 32];
  __shared__ unsigned long long s_prefix;
  __shared__ uint32_t s_chunk;
  const int tid = threadIdx.x;
  if (tid == 0) s_chunk = atomicAdd(&small[kSmScanCounter], 1u);
  for (int i = tid; i < kMaxTilePasses * 256; i += kScanThreads) (&s_hist[0][0])[i] = 0u;
  __syncthreads();
  const int64_t chunk = s_chunk;
  const int64_t nchunks = (n + kScanChunk - 1) / kScanChunk;
  const int64_t base = chunk * kScanChunk;
  const float4* q0 = reinterpret_cast<const float4*>(proj);
  const float4* q1 = q0 + n;
#pragma unroll
  for (int j = 0; j < kScanItems; ++j) {
    const int li = j * kScanThreads + tid;
    const int64_t i = base + li;
    uint32_t cnt = 0, rect = 0, width = 1, g = 0;
    if (i < n && skey[i] != kCulledKey) {
      g = sidx[i];
      const int r = __float_as_int(__ldg(&q1[g].w));
      const float4 a = __ldg(&q0[g]);
      const int fu = (int)floorf(fminf(fmaxf(a.x, -1e9f), 1e9f));
      const int fv = (int)floorf(fminf(fmaxf(a.y, -1e9f), 1e9f));
      const int x0 = min(max((fu - r) >> 4, 0), k.Tx), x1 = min(max(((fu + r) >> 4) + 1, 0), k.Tx);
      const int y0 = min(max((fv - r) >> 4, 0), k.Ty), y1 = min(max(((fv + r) >> 4) + 1, 0), k.Ty);
      if (r > 0 && x0 < x1 && y0 < y1) {
        cnt = (uint32_t)((x1 - x0) * (y1 - y0));
        rect = (uint32_t)x0 | ((uint32_t)y0 << 16);
        width = (uint32_t)(x1 - x0);
      }
    }
    s_items[li] = cnt;
    s_rect[li] = rect;
    s_width[li] = width;
    s_rcpw[li] = 1.0f / (float)width;
    s_gauss[li] = g;
  }
  __syncthreads();
  // blocked scan: thread t owns items t*kScanItems .. +kScanItems-1
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
    if (to) flag_status(count, gs::kStatusTimeout);
    s_prefix = excl;
    if (chunk == nchunks - 1) {
      const int64_t M = (int64_t)(excl + total);
      count[0] = M;
      if (M > cap) flag_status(count, gs::kStatusCapacity);
    }
  }
  __syncthreads();
  // Cooperative, coalesced write of this chunk's instances, one window of kWin output slots
  // at a time: every item whose run meets the window marks its first slot there with its
  // index + 1, and an inclusive max-scan over the window turns the marks into the owner of
  // every slot (items are in offset order).
  const int64_t out0 = (int64_t)s_prefix;
  for (uint32_t w0 = 0; w0 < total; w0 += kWin) {
    const uint32_t wn = min((uint32_t)kWin, total - w0);
    for (int i = tid; i < kWin; i += kScanThreads) s_owner[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kScanItems; ++j) {
      const int li = tid * kScanItems + j;
      const uint32_t off = s_items[li], c = v[j];
      if (c > 0 && off < w0 + wn && off + c > w0) s_owner[max(off, w0) - w0] = (uint32_t)li + 1u;
    }
    __syncthreads();
    {  // inclusive max-scan of s_owner[0 .. kWin): kWinPer consecutive slots per thread
      uint32_t run = 0;
#pragma unroll
      for (int e = 0; e < kWinPer; ++e) run = max(run, s_owner[tid * kWinPer + e]);
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = max(incl, y);
      }
      if (lane == 31) s_warp[warp] = incl;
      __syncthreads();
      uint32_t carry = 0;
      for (int w = 0; w < warp; ++w) carry = max(carry, s_warp[w]);
      uint32_t prev = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) prev = 0u;
      run = max(carry, prev);
#pragma unroll
      for (int e = 0; e < kWinPer; ++e) {
        run = max(run, s_owner[tid * kWinPer + e]);
        s_owner[tid * kWinPer + e] = run;
      }
    }
    __syncthreads();
    for (uint32_t q = tid; q < wn; q += kScanThreads) {
      const uint32_t li = s_owner[q] - 1u;
      const uint32_t j = w0 + q - s_items[li];  // index of the tile inside the item's rectangle
      const uint32_t w = s_width[li];
      // j / w from a float estimate, corrected once (|error| <= 1 for j < 2^24)
      uint32_t row = (uint32_t)__fmul_rz((float)j, s_rcpw[li]);
      int rem = (int)j - (int)(row * w);
      if (rem < 0) { --row; rem += (int)w; }
      if (rem >= (int)w) { ++row; rem -= (int)w; }
      const uint32_t rect = s_rect[li];
      const uint32_t tile = ((rect >> 16) + row) * (uint32_t)k.Tx + (rect & 0xffffu) + (uint32_t)rem;
      const int64_t o = out0 + w0 + q;
      if (o < cap) {
        tkey[o] = tile;
        tval[o] = s_gauss[li];
      }
      for (int pp = 0; pp < tpasses; ++pp) atomicAdd(&s_hist[pp][(tile >> (8 * pp)) & 255u], 1u);
    }
    __syncthreads();
  }
  for (int i = tid; i < tpasses * 256; i += kScanThreads) {
    const uint32_t c = (&s_hist[0][0])[i];
    if (c) atomicAdd(&small[kSmHist + kDepthPasses * 256 + i], c);
  }
}

// ------------------------------------------------------------------ keys, values, ranges
__global__ void __launch_bounds__(256) k_finalize(const float* __restrict__ proj, const uint32_t* __restrict__ tkey,
                                                   const uint32_t* __restrict__ tval, int64_t cap,
                                                   uint64_t* __restrict__ keys, uint32_t* __restrict__ vals,
                                                   uint32_t* __restrict__ ranges, const int64_t* count) {
  if (count[1] != 0) return;
  const float4* q0 = reinterpret_cast<const float4*>(proj);
  const int64_t M = min(count[0], cap);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < M; i += stride) {
    const uint32_t t = tkey[i], g = tval[i];
    keys[i] = ((uint64_t)t << 32) | __float_as_uint(__ldg(&q0[g].z));
    vals[i] = g;
    if (i == 0 || tkey[i - 1] != t) ranges[2 * (int64_t)t] = (uint32_t)i;
    if (i == M - 1 || tkey[i + 1] != t) ranges[2 * (int64_t)t + 1] = (uint32_t)(i + 1);
  }
}

template <int ITEMS>
int sort_blocks_per_sm() {
  static int cached = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (cached < 0) {
    int b = 0;
    const int bytes = (int)sizeof(SortSmem<ITEMS>);
    cudaFuncSetAttribute(k_onesweep<ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_onesweep<ITEMS>, kSortThreads, bytes) != cudaSuccess ||
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
  return carve(nullptr, nullptr, n, capacity, tile_passes(k));
}

extern "C" gs_status gs_bin_sort(const float* proj, int64_t n, const gs_camera* cam, void* workspace,
                                 size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                                 uint32_t* ranges, int64_t* count, int64_t* count_host, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  if (n < 0 || n >= (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: bad n");
  if (capacity < 0 || capacity >= (int64_t(1) << 30))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: capacity must be in [0, 2^30)");
  if (!count || !ranges || (n > 0 && !proj) || (capacity > 0 && (!keys || !vals)) || !workspace)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: NULL pointer");
  if ((proj && !gs::aligned16(proj)) || !gs::aligned8(count) || (keys && !gs::aligned8(keys)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: misaligned pointer");
  const gs::Cam k = gs::make_cam(*cam);
  const int tpasses = tile_passes(k);
  if (tpasses > kMaxTilePasses) return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: too many tiles");
  const size_t need = carve(nullptr, nullptr, n, capacity, tpasses);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: workspace %zu bytes < %zu needed", workspace_bytes, need);
  Workspace w;
  carve(&w, reinterpret_cast<char*>(workspace), n, capacity, tpasses);
  cudaStream_t st = gs::as_stream(stream);
  const int64_t T = (int64_t)k.Tx * k.Ty;
  const int64_t limit = gs::wait_limit();
  const int drop = gs::take_drop_publish();

  if (cudaMemsetAsync(count, 0, 2 * sizeof(int64_t), st) != cudaSuccess ||
      cudaMemsetAsync(w.small, 0, sizeof(uint32_t) * kSmWords, st) != cudaSuccess ||
      cudaMemsetAsync(ranges, 0, sizeof(uint32_t) * 2 * T, st) != cudaSuccess)
    return gs::check_launch("gs_bin_sort memset");
  if (n > 0) {
    const int64_t chunks = (n + kScanChunk - 1) / kScanChunk;
    if (cudaMemsetAsync(w.scan_state, 0, sizeof(unsigned long long) * chunks, st) != cudaSuccess)
      return gs::check_launch("gs_bin_sort memset");
    const int sms = gs::num_sms();
    // 1. Gaussians by (depth, index): 4 stable passes over 32-bit depth keys
    const int64_t lb_tile_words = (int64_t)tpasses * sort_tiles<kTileItems>(capacity) * 256;
    k_depth_init<<<sms * 4, 256, 0, st>>>(proj, n, w.dkey[0], w.didx[0], w.small, w.lb_depth, w.lb_tile,
                                          lb_tile_words);
    k_digit_scan<<<1, 256, 0, st>>>(w.small, 0, kDepthPasses, count);
    const int grid_d = (int)std::min<int64_t>(sms * sort_blocks_per_sm<kDepthItems>(), sort_tiles<kDepthItems>(n));
    for (int p = 0; p < kDepthPasses; ++p) {
      k_onesweep<kDepthItems><<<grid_d, kSortThreads, sizeof(SortSmem<kDepthItems>), st>>>(
          w.dkey[p & 1], w.didx[p & 1], w.dkey[(p + 1) & 1], w.didx[(p + 1) & 1], n, n, 8 * p, p, w.small,
          w.lb_depth + (size_t)p * sort_tiles<kDepthItems>(n) * 256, count, limit, p == 0 ? drop : 0);
    }
    if (gs_status s = gs::check_launch("gs_bin_sort depth sort")) return s;
    // 2. (tile, index) pairs in depth order, with their tile-digit histograms
    k_scan_dup<<<(unsigned)chunks, kScanThreads, 0, st>>>(proj, n, w.dkey[0], w.didx[0], k, tpasses, w.tkey[0],
                                                           w.tval[0], capacity, w.scan_state, w.small, count, limit);
    if (gs_status s = gs::check_launch("gs_bin_sort scan")) return s;
    // 3. stable sort of the pairs by tile id
    k_digit_scan<<<1, 256, 0, st>>>(w.small, kDepthPasses, tpasses, count);
    const int grid_t = sms * sort_blocks_per_sm<kTileItems>();
    for (int p = 0; p < tpasses; ++p) {
      k_onesweep<kTileItems><<<grid_t, kSortThreads, sizeof(SortSmem<kTileItems>), st>>>(
          w.tkey[p & 1], w.tval[p & 1], w.tkey[(p + 1) & 1], w.tval[(p + 1) & 1], -1, capacity, 8 * p,
          kDepthPasses + p, w.small, w.lb_tile + (size_t)p * sort_tiles<kTileItems>(capacity) * 256, count, limit, 0);
    }
    if (gs_status s = gs::check_launch("gs_bin_sort tile sort")) return s;
    k_finalize<<<sms * 8, 256, 0, st>>>(proj, w.tkey[tpasses & 1], w.tval[tpasses & 1], capacity, keys, vals, ranges,
                                        count);
    if (gs_status s = gs::check_launch("gs_bin_sort finalize")) return s;
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
