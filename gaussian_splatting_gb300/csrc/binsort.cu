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
//   k_sort_init   zeroes the status words, the small block, the staged ranges and the
//                 caller's ranges of every view of a group (one launch instead of memsets).
//   k_depth_sort  all stable 8-bit passes of the depth sorts of up to 8 views in one
//                 cooperative launch (a group of CTAs per view, so the views' latency-bound
//                 phases overlap).  Each pass counts digits per radix tile, scans the counts
//                 per digit over the tiles (the column sums are the digit totals), then ranks
//                 every tile in shared memory and writes digit-contiguous runs at the digit's
//                 base (an exclusive scan of the totals) plus its column offset; grid
//                 barriers (per view) separate the phases.  Phase 0 makes the depth keys
//                 and an 8-byte tile-rectangle record per visible Gaussian; pass 0 leaves the
//                 culled ones out, so the later passes move only the visible keys.  After the
//                 passes the same launch runs the tiles-touched scan over the sorted visible
//                 Gaussians (each CTA a contiguous run of chunks: their sums, the CTAs'
//                 totals, then each chunk's
//                 records: first slot, rectangle, index; and for every radix tile of the tile
//                 sort the Gaussian holding its first slot).
//   k_tile_sort   the same passes for one view's instances by tile id: the first pass
//                 generates its (tile, index) pairs from the scan's records instead of reading
//                 them, the last writes the caller's values (and 64-bit keys if asked for) and
//                 the sorted tile ids, from whose boundaries a final phase stages the ranges.
//   k_publish_ranges  copies each view's staged ranges to the caller's array if nothing failed.
// Every device-side wait is bounded (gs_debug_set_wait_limit); on expiry the kernel sets
// status bit 2 in count[1] and carries on, so nothing can hang.
#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

constexpr int kScanChunk = 1024;  // sorted Gaussians per chunk of the tiles-touched scan
constexpr int kMaxScanCtas = 4096;  // CTAs per view of a depth-sort launch (their scan totals)
// CTAs per view at least (as many as resident allow), however few the radix tiles: phase B
// scans 256 digit columns, one CTA each at a time
constexpr int64_t kMinSortCtas = 64;

constexpr int kSortThreads = 256;
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kDepthItems = 4;    // depth passes: 1024 keys per radix tile (N is modest)
constexpr int64_t kWideDepthN = 2000000;  // from this many Gaussians on, 3072 keys per radix tile
#ifndef GS_TILE_ITEMS
#define GS_TILE_ITEMS 12
#endif
#ifndef GS_SORT_MIN_BLOCKS
#define GS_SORT_MIN_BLOCKS 4
#endif
constexpr int kTileItems = GS_TILE_ITEMS;  // tile passes: 3072 keys per radix tile (M is large)
constexpr int kSlice = kSortThreads * kTileItems;  // instances per generated radix tile
constexpr int kDepthPasses = 4;
constexpr int kMaxSortViews = 8;  // views per sort launch
// views whose tile sorts share a launch: as many as have their own capacity-sized ping-pong
// buffers within this budget (at least one, at most kMaxSortViews)
#ifndef GS_TILE_BUDGET_MB
#define GS_TILE_BUDGET_MB 1024
#endif
constexpr double kTileBudgetBytes = GS_TILE_BUDGET_MB * 1024.0 * 1024.0;
constexpr int kMaxTilePasses = 4;
constexpr int kSlots = kDepthPasses + kMaxTilePasses;  // digit histogram / base slots

constexpr uint32_t kCulledKey = 0xFFFFFFFFu;

// layout of the small, memset-cleared block of the workspace (32-bit words)
constexpr int kSmBarrier = 1;        // one arrival counter per sort (depth, tile)
constexpr int kSmVisible = 3;        // the depth sort's count of visible Gaussians, for the tile sort
constexpr int kSmTileCtr = 4;        // phase C's radix-tile counters: [sort][pass], kMaxTilePasses each
constexpr int kSmHist = 32;          // kSlots * 256 digit totals (the column sums of phase B)
static_assert(kDepthPasses <= kMaxTilePasses && kSmTileCtr + 2 * kMaxTilePasses <= kSmHist, "small-block layout");
constexpr int kSmWords = kSmHist + kSlots * 256;

struct Workspace {
  uint32_t* tkey[2];               // instance tile ids, ping-pong
  uint32_t* tval[2];               // instance Gaussian indices, ping-pong
  uint32_t* dkey[2];
  uint32_t* didx[2];
  unsigned long long* cta_tot;     // per CTA of the view's depth sort: tiles touched by its chunks
  uint32_t* hist_depth;            // [256][radix tiles of the depth sort]
  uint32_t* hist_tile;             // [256][radix tiles of the tile sort]
  uint2* rrec;                     // per Gaussian (index order): (x0 | y0 << 16, w | h << 16)
  uint32_t* rstage;                // tile ranges, published to the caller only on success
  uint32_t* slice_first;           // per output slice of kSlice slots: the item holding its first slot
  uint4* grec;                     // per depth-ordered Gaussian: (slot, x0 | y0 << 16, w | h << 16, index)
  uint32_t* small;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
template <int ITEMS>
__host__ __device__ inline int64_t sort_tiles(int64_t m) {
  constexpr int kTile = kSortThreads * ITEMS;
  return (m + kTile - 1) / kTile;
}

// Row length of a [256][radix tiles] digit-count table: the tile count rounded up to a multiple
// of four, so that every digit's row starts on a 16-byte boundary (phase B reads it as uint4).
inline int64_t hist_cols(int64_t tiles) { return (tiles + 3) / 4 * 4; }

int tile_bits(int64_t T) {
  int b = 0;
  while ((int64_t(1) << b) < T) ++b;
  return b;
}

int tile_passes(const gs::Cam& k) { return std::max(1, (tile_bits((int64_t)k.Tx * k.Ty) + 7) / 8); }

// Workspace layout: `tile_slots` sets of tile-sort buffers (capacity-sized; view v uses set
// v % tile_slots, the views of one tile-sort launch having sets of their own), then per view
// the depth-sort buffers and the scan's records.  w (if not NULL) receives `views` entries.
size_t carve(Workspace* w, char* base, int views, int64_t n, int64_t cap, int64_t n_tiles, int tile_slots) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align256(std::max<size_t>(bytes, 1));
    return p;
  };
  char* tk[kMaxSortViews][5];
  for (int t = 0; t < tile_slots; ++t) {
    for (int j = 0; j < 4; ++j) tk[t][j] = take(sizeof(uint32_t) * (size_t)cap);
    tk[t][4] = take(sizeof(uint32_t) * 256 * (size_t)hist_cols(sort_tiles<kTileItems>(cap)));
  }
  for (int v = 0; v < views; ++v) {
    char* dk0 = take(sizeof(uint32_t) * (size_t)n);
    char* dk1 = take(sizeof(uint32_t) * (size_t)n);
    char* di0 = take(sizeof(uint32_t) * (size_t)n);
    char* di1 = take(sizeof(uint32_t) * (size_t)n);
    char* ss = take(sizeof(unsigned long long) * (size_t)kMaxScanCtas);
    char* lbd = take(sizeof(uint32_t) * 256 * (size_t)hist_cols(sort_tiles<kDepthItems>(n)));
    char* rr = take(sizeof(uint2) * (size_t)n);
    char* rs = take(sizeof(uint32_t) * 2 * (size_t)n_tiles);
    char* go = take(sizeof(uint32_t) * (size_t)((cap + kSlice - 1) / kSlice));
    char* gr4 = take(sizeof(uint4) * (size_t)n);
    char* sm = take(sizeof(uint32_t) * kSmWords);
    if (w) {
      Workspace& x = w[v];
      char* const* t = tk[v % tile_slots];
      x.tkey[0] = reinterpret_cast<uint32_t*>(t[0]);
      x.tkey[1] = reinterpret_cast<uint32_t*>(t[1]);
      x.tval[0] = reinterpret_cast<uint32_t*>(t[2]);
      x.tval[1] = reinterpret_cast<uint32_t*>(t[3]);
      x.hist_tile = reinterpret_cast<uint32_t*>(t[4]);
      x.dkey[0] = reinterpret_cast<uint32_t*>(dk0);
      x.dkey[1] = reinterpret_cast<uint32_t*>(dk1);
      x.didx[0] = reinterpret_cast<uint32_t*>(di0);
      x.didx[1] = reinterpret_cast<uint32_t*>(di1);
      x.cta_tot = reinterpret_cast<unsigned long long*>(ss);
      x.hist_depth = reinterpret_cast<uint32_t*>(lbd);
      x.rrec = reinterpret_cast<uint2*>(rr);
      x.rstage = reinterpret_cast<uint32_t*>(rs);
      x.slice_first = reinterpret_cast<uint32_t*>(go);
      x.grec = reinterpret_cast<uint4*>(gr4);
      x.small = reinterpret_cast<uint32_t*>(sm);
    }
  }
  return off;
}

__device__ __forceinline__ void flag_status(int64_t* count, int64_t bits) {
  atomicOr(reinterpret_cast<unsigned long long*>(&count[1]), (unsigned long long)bits);
}

// ------------------------------------------------------------------ stable radix sort
// One cooperative launch runs every pass of a sort.  Each pass is reduce-then-scan over
// radix tiles of kSortThreads * ITEMS keys, with grid-wide barriers between the phases:
//   A  every radix tile's digit counts -> hist[digit][tile];
//   B  per digit, the exclusive scan of its counts over the tiles plus the digit's global
//      base (digit sums are known beforehand) -> the tile's first output slot for it;
//   C  every tile ranks its keys stably (warp match-any ranking in shared memory),
//      scatters them through shared memory and writes digit-contiguous runs.
// CTA b takes tiles b, b + G, ... in A and C (a tile's offsets no longer depend on the
// order tiles are processed in), so no CTA ever waits on another inside a phase.
template <int ITEMS>
struct SortSmem {
  uint32_t keys[kSortThreads * ITEMS];
  uint32_t vals[kSortThreads * ITEMS];
  uint32_t whist[kSortWarps][256];
  uint32_t peer[kSortWarps][256];  // all zero between uses
  uint32_t tstart[256];
  uint32_t gbase[256];
  uint32_t dbase[256];  // the pass's digit bases
  uint32_t wsum[kSortWarps];
  uint32_t full;    // first tile pass, counts: full cycles of 256 digits
  uint32_t nxt[2];  // phase C: the radix tiles taken from the counter (current, next)
  uint32_t total;   // the pass's key count (sum of the digit totals)
  uint32_t tvalid;  // phase C: keys of the current radix tile that take part in the pass
  int fail;
};

// Pass 0 of the tile sort generates its pairs: they are the tile instances in depth order,
// slot o belonging to the depth-ordered Gaussian whose run [offset, offset + tiles) holds o.
// A radix tile is one slice of the scan's slice_first table; the Gaussians starting inside it
// mark their first slot, an inclusive max-scan turns the marks into each slot's owner, and
// the owner's rectangle record gives the tile id.
struct GenSource {
  const uint32_t* slice_first;  // per radix tile: the Gaussian holding its first slot
  const uint4* grec;            // per depth-ordered visible Gaussian: (offset, x0 | y0 << 16, w | h << 16, index)
  int Tx;
};

struct RadixJob {
  uint32_t* key[2];     // ping-pong: pass p reads key[p & 1] and writes key[(p + 1) & 1]
  uint32_t* val[2];
  int64_t n_host;       // >= 0: sort n_host keys; < 0: min(count[0], cap)
  int64_t cap;
  int passes;
  int slot0;            // digit-base slot of pass 0 in the small block
  int sort_id;          // selects the barrier word and tile counters in the small block
  uint32_t* hist;       // [256][hist_stride]
  int64_t hist_stride;  // radix tiles per digit row
  uint32_t* small;
  int64_t* count;
  int64_t limit;
  int drop_arrival;     // test hook: CTA 0 never arrives at the first barrier
  GenSource gen;        // tile sort only (gen.grec != nullptr): pass 0 generates its pairs
  const float4* q0;     // tile sort only: the last pass writes (key << 32 | depth bits of
  uint64_t* keys64;     // Gaussian value) to keys64 and the values to vals_out
  uint32_t* vals_out;
  // depth sort only: phase 0 makes the keys and the rectangle records from the projection
  const float* proj;
  int Tx, Ty;
  uint2* rrec;          // per Gaussian, index order: (x0 | y0 << 16, w | h << 16); 0 if culled
  // depth sort only, after the last pass: the tiles-touched scan over the depth-sorted
  // Gaussians
  unsigned long long* cta_tot;    // per CTA of the job: tiles touched by its scan chunks
  uint4* grec;          // per sorted Gaussian: (first slot, x0 | y0 << 16, w | h << 16, index)
  uint32_t* slice_first;  // per radix tile of the tile sort: the Gaussian holding its first slot
  int64_t tcap;         // instance capacity
  // tile sort only: after the last pass, the staged ranges from the sorted tile ids (zeroed by
  // the host, published to the caller if nothing failed)
  uint32_t* rstage;
};

// The sort jobs of one launch (kernel parameter space: 8 jobs stay under 4 KB).
struct RadixBatch {
  RadixJob job[kMaxSortViews];
  int views;
};
static_assert(sizeof(RadixBatch) <= 4000, "depth-sort jobs must fit the kernel parameter space");
static_assert(sizeof(RadixJob) % 4 == 0, "jobs are copied as 32-bit words");

// Grid-wide barrier on a monotonically increasing arrival counter.  Bounded: after `limit`
// polls, or once another CTA has reported a failure, it sets/keeps status bit 2 and returns
// false so the caller can leave.
template <int ITEMS>
__device__ bool grid_barrier(SortSmem<ITEMS>& S, const RadixJob& J, uint32_t target, bool arrive) {
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* bar = J.small + kSmBarrier + J.sort_id;
    int fail = 0;
    if (arrive) {
      __threadfence();
      atomicAdd(bar, 1u);
    }
    for (int64_t it = 0; ld_acquire_u32(bar) < target; ++it) {
      if (it >= J.limit) {
        flag_status(J.count, gs::kStatusTimeout);
        fail = 1;
        break;
      }
      if ((it & 63) == 63 && ld_acquire_u64(reinterpret_cast<const unsigned long long*>(&J.count[1])) != 0) {
        fail = 1;
        break;
      }
      if (it > 8) __nanosleep(32);
    }
    __threadfence();
    S.fail = fail;
  }
  __syncthreads();
  return S.fail == 0;
}

// Row and column of tile j of a rectangle w tiles wide (w >= 1): a float estimate of j / w,
// within 1 of the quotient (its relative error is about 2^-21 and quotients stay below 2^16),
// corrected by one step either way.
__device__ __forceinline__ uint32_t rect_row(uint32_t j, uint32_t w, uint32_t& col) {
  uint32_t row = (uint32_t)__fmul_rz((float)j, __fdividef(1.f, (float)w));
  int rem = (int)j - (int)(row * w);
  if (rem < 0) { --row; rem += (int)w; }
  if (rem >= (int)w) { ++row; rem -= (int)w; }
  col = (uint32_t)rem;
  return row;
}

// 32-bit words of radix tile `tile` of an M-word array, warp-striped: item i of lane l of warp
// w is slot w * ITEMS * 32 + i * 32 + l; slots past M read nothing and get 0.
template <int ITEMS>
__device__ __forceinline__ void load_words(const uint32_t* in, int64_t tile, int64_t M, uint32_t (&x)[ITEMS]) {
  constexpr int kTile = kSortThreads * ITEMS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t base = tile * kTile;
  const int64_t nvalid = min((int64_t)kTile, M - base);
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int li = warp * (ITEMS * 32) + i * 32 + lane;
    x[i] = li < nvalid ? __ldcg(&in[base + li]) : 0u;
  }
}

// The keys (tile ids) and values (Gaussian indices) of radix tile `tile` of the first tile
// pass, generated in the warp-striped order of load_words.  Slots past nvalid get key
// 0xFFFFFFFF.  The records of the first Gaussians from `first` on are kept in S.whist (free
// until the ranking; the caller clears it afterwards), so most slots read their owner's
// record from shared memory.
template <int ITEMS>
__device__ __forceinline__ void gen_tile(SortSmem<ITEMS>& S, const RadixJob& J, int64_t tile, int64_t base,
                                         int nvalid, uint32_t (&k)[ITEMS], uint32_t (&v)[ITEMS]) {
  constexpr int kTile = kSortThreads * ITEMS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wbase = warp * (ITEMS * 32);
  const bool full = nvalid == kTile;
  uint32_t* own = S.keys;  // free until the scatter
  uint4* rc = reinterpret_cast<uint4*>(&S.whist[0][0]);
  constexpr uint32_t kRecCache = sizeof(S.whist) / sizeof(uint4);
  const GenSource& G = J.gen;
  const int64_t gn = __ldg(&J.small[kSmVisible]);  // depth-ordered visible Gaussians (previous launch)
  const int64_t first = (int64_t)__ldg(&G.slice_first[tile]);
  for (int i = tid; i < kTile; i += kSortThreads) own[i] = 0u;
  __syncthreads();
  // Offsets rise with e, so the Gaussians starting inside the tile are a prefix of those
  // after `first`; a Gaussian with no tiles shares its offset with the next one, whence the
  // max (the last Gaussian at an offset is the one that owns it).
  const uint32_t end = (uint32_t)(base + nvalid);
  for (int e0 = 0;; e0 += kSortThreads) {
    const int64_t it = first + e0 + tid;
    const uint4 r = it < gn ? __ldg(&G.grec[it]) : make_uint4(0xFFFFFFFFu, 0u, 0u, 0u);
    const uint32_t off = r.x;
    if ((uint32_t)(e0 + tid) < kRecCache) rc[e0 + tid] = r;
    const bool first_item = e0 + tid == 0;
    const bool in = first_item || off < end;
    if (in && it < gn) atomicMax(&own[first_item ? 0u : off - (uint32_t)base], (uint32_t)(e0 + tid) + 1u);
    if (!__syncthreads_or(!first_item && off < end)) break;
  }
  {  // inclusive max-scan of the marks, ITEMS consecutive slots per thread
    uint32_t tmax = 0;
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) tmax = max(tmax, own[tid * ITEMS + e]);
    uint32_t incl = tmax;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl = max(incl, y);
    }
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    uint32_t carry = 0;
    for (int w = 0; w < warp; ++w) carry = max(carry, S.wsum[w]);
    uint32_t prev = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) prev = 0u;
    uint32_t r = max(carry, prev);
#pragma unroll
    for (int e = 0; e < ITEMS; ++e) {
      r = max(r, own[tid * ITEMS + e]);
      own[tid * ITEMS + e] = r;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int li = wbase + i * 32 + lane;
    const uint32_t o = own[li];
    if ((full || li < nvalid) && o != 0u && first + o - 1u < gn) {
      const uint32_t e = o - 1u;
      const uint4 rec = e < kRecCache ? rc[e] : __ldg(&G.grec[first + e]);
      uint32_t col;
      const uint32_t row = rect_row((uint32_t)(base + li) - rec.x, max(rec.z & 0xffffu, 1u), col);
      k[i] = ((rec.y >> 16) + row) * (uint32_t)G.Tx + (rec.y & 0xffffu) + col;
      v[i] = rec.w;
    } else {
      k[i] = 0xFFFFFFFFu;
      v[i] = 0u;
    }
  }
  __syncthreads();  // own[] (= S.keys) is reused by the caller
}

// Low-byte digit counts of the tile ids that radix tile `tile` of the first tile pass
// generates, without generating them: the tile holds whole or partial rectangle rows of the
// Gaussians starting in it (and of the one holding its first slot); a row segment is a run
// of consecutive tile ids, i.e. a cyclic run of digits, added to a difference array (every
// full cycle of 256 adds one to every digit).  Leaves the counts in S.tstart.
template <int ITEMS>
__device__ __forceinline__ void gen_digit_counts(SortSmem<ITEMS>& S, const RadixJob& J, int64_t tile, int64_t base,
                                                 int nvalid, int64_t M) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const GenSource& G = J.gen;
  const int64_t gn = __ldg(&J.small[kSmVisible]);  // depth-ordered visible Gaussians (previous launch)
  uint32_t* diff = S.tstart;  // zeroed by the caller
  if (tid == 0) S.full = 0u;
  __syncthreads();
  const int64_t first = (int64_t)__ldg(&G.slice_first[tile]);
  const uint32_t lo = (uint32_t)base, end = (uint32_t)(base + nvalid);
  for (int e0 = 0;; e0 += kSortThreads) {
    const int64_t it = first + e0 + tid;
    const uint4 rec = it < gn ? __ldg(&G.grec[it]) : make_uint4(0xFFFFFFFFu, 0u, 0u, 0u);
    const uint32_t off = rec.x;
    // the next Gaussian's first slot: the next lane's record (one load per warp for lane 31)
    uint32_t next = __shfl_down_sync(0xffffffffu, off, 1);
    if (lane == 31 && it + 1 < gn) next = __ldg(&G.grec[it + 1]).x;
    if (it + 1 >= gn) next = (uint32_t)M;
    bool more = false;
    if (it < gn) {
      more = off < end;
      if (more || e0 + tid == 0) {
        const uint32_t s_lo = max(off, lo), s_hi = min(next, end);
        const uint32_t w = max(rec.z & 0xffffu, 1u);
        if (s_lo < s_hi) {
          const uint32_t x0 = rec.y & 0xffffu, y0 = rec.y >> 16;
          uint32_t c0, c1;
          const uint32_t r0 = rect_row(s_lo - off, w, c0), r1 = rect_row(s_hi - 1u - off, w, c1);
          for (uint32_t r = r0; r <= r1; ++r) {
            const uint32_t j_lo = r == r0 ? c0 : 0u;
            const uint32_t j_hi = r == r1 ? c1 : w - 1u;
            const uint32_t t_lo = (y0 + r) * (uint32_t)G.Tx + x0 + j_lo;
            const uint32_t len = j_hi - j_lo + 1u;
            if (len >> 8) atomicAdd(&S.full, len >> 8);
            const uint32_t rem = len & 255u, a = t_lo & 255u;
            if (rem) {
              atomicAdd(&diff[a], 1u);
              if (a + rem < 256u) atomicAdd(&diff[a + rem], 0xFFFFFFFFu);
              else if (a + rem > 256u) {  // wraps: [a, 256) and [0, a + rem - 256)
                atomicAdd(&diff[0], 1u);
                atomicAdd(&diff[a + rem - 256u], 0xFFFFFFFFu);
              }
            }
          }
        }
      }
    }
    if (!__syncthreads_or(more)) break;
  }
  // counts = inclusive prefix of the difference array (one digit per thread) + full cycles
  const uint32_t dv = diff[tid];
  uint32_t incl = dv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) S.wsum[warp] = incl;
  __syncthreads();
  uint32_t woff = 0;
  for (int w2 = 0; w2 < warp; ++w2) woff += S.wsum[w2];
  const uint32_t cnt = woff + incl + S.full;
  __syncthreads();
  diff[tid] = cnt;
  __syncthreads();
}

// Depth sort, phase 0 (replaces phase A of pass 0): radix tile by radix tile, the depth key of
// every Gaussian (float bits of z; 0xFFFFFFFF if culled), its index, the tile-rectangle record
// of every visible one and the tile's pass-0 digit counts of the visible keys only: pass 0
// drops the culled Gaussians, so the later passes and the scan see only the visible ones.
template <int ITEMS>
__device__ __forceinline__ void depth_phase0(SortSmem<ITEMS>& S, const RadixJob& J, int64_t n, int64_t ntiles,
                                             uint32_t G, uint32_t bid) {
  constexpr int kTile = kSortThreads * ITEMS;
  const int tid = threadIdx.x;
  const float4* q0 = reinterpret_cast<const float4*>(J.proj);
  const float4* q1 = q0 + n;
  for (int64_t tile = bid; tile < ntiles; tile += G) {
    for (int i = tid; i < 256; i += kSortThreads) S.tstart[i] = 0u;
    __syncthreads();
    for (int j = tid; j < kTile; j += kSortThreads) {
      const int64_t i = tile * kTile + j;
      if (i >= n) break;
      const int r = __float_as_int(__ldg(&q1[i].w));
      const float4 a = __ldg(&q0[i]);
      uint32_t key = kCulledKey;
      uint2 rec = make_uint2(0u, 0u);
      if (r > 0) {
        const int fu = (int)floorf(fminf(fmaxf(a.x, -1e9f), 1e9f));
        const int fv = (int)floorf(fminf(fmaxf(a.y, -1e9f), 1e9f));
        const int x0 = min(max((fu - r) >> 4, 0), J.Tx), x1 = min(max(((fu + r) >> 4) + 1, 0), J.Tx);
        const int y0 = min(max((fv - r) >> 4, 0), J.Ty), y1 = min(max(((fv + r) >> 4) + 1, 0), J.Ty);
        key = __float_as_uint(a.z);  // finite and positive: never the culled key
        if (x0 < x1 && y0 < y1)
          rec = make_uint2((uint32_t)x0 | ((uint32_t)y0 << 16), (uint32_t)(x1 - x0) | ((uint32_t)(y1 - y0) << 16));
        J.rrec[i] = rec;
        atomicAdd(&S.tstart[key & 255u], 1u);
      }
      J.key[0][i] = key;
      J.val[0][i] = (uint32_t)i;
    }
    __syncthreads();
    J.hist[(int64_t)tid * J.hist_stride + tile] = S.tstart[tid];
    __syncthreads();
  }
}

// Tiles touched by Gaussian g (from its rectangle record) and its scan record (first slot
// left 0; z = width | height << 16).
__device__ __forceinline__ uint32_t touched(const RadixJob& J, uint32_t g, uint4& rec) {
  const uint2 r = __ldcg(&J.rrec[g]);  // written by other CTAs of this launch
  rec = make_uint4(0u, r.x, r.y, g);
  return (r.y & 0xffffu) * (r.y >> 16);
}

// After the depth passes: the tiles-touched scan over the n sorted visible Gaussians, in chunks
// of kScanChunk; CTA b owns a contiguous run of chunks.  S1: every sorted Gaussian's record
// (gathered once, by index, from the rectangle records) and the sum of every chunk; the CTA's
// total.  S3: the CTA's first slot (the totals of the CTAs before it), then every chunk's
// first slots in order, the records read back and completed, and the first Gaussian of every
// radix tile of the tile sort; the last CTA's end is M.  Returns false if a barrier failed.
template <int ITEMS>
__device__ bool depth_scan(SortSmem<ITEMS>& S, const RadixJob& J, int64_t n, uint32_t G, uint32_t bid,
                           uint32_t& nbar) {
  constexpr int kPer = kScanChunk / kSortThreads;  // 4 consecutive Gaussians per thread
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nchunks = (n + kScanChunk - 1) / kScanChunk;
  const int64_t per = (nchunks + G - 1) / G;
  const int64_t c_begin = min((int64_t)bid * per, nchunks), c_end = min(c_begin + per, nchunks);
  const uint32_t* sidx = J.val[kDepthPasses & 1];
  unsigned long long* wsum64 = reinterpret_cast<unsigned long long*>(S.gbase);  // free in these phases
  // S1: records and the CTA's total (a thread keeps its kPer Gaussians of every chunk for S3;
  // no barrier per chunk, two chunks' gathers in flight)
  unsigned long long tsum = 0;
#pragma unroll 2
  for (int64_t c = c_begin; c < c_end; ++c) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t i = c * kScanChunk + tid * kPer + j;
      if (i < n) {
        uint4 rec;
        tsum += touched(J, __ldcg(&sidx[i]), rec);
        J.grec[i] = rec;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
  if (lane == 0) wsum64[warp] = tsum;
  __syncthreads();
  unsigned long long run = 0;
  for (int w = 0; w < kSortWarps; ++w) run += wsum64[w];
  if (tid == 0) J.cta_tot[bid] = run;
  if (!grid_barrier(S, J, ++nbar * G, true)) return false;
  // S3: the CTA's first slot, then its chunks in order
  unsigned long long part = 0;
  for (uint32_t b2 = tid; b2 < bid; b2 += kSortThreads) part += __ldcg(&J.cta_tot[b2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  __syncthreads();
  if (lane == 0) wsum64[warp] = part;
  __syncthreads();
  unsigned long long prefix = 0;
  for (int w = 0; w < kSortWarps; ++w) prefix += wsum64[w];
  if (bid == G - 1 && tid == 0) {
    const int64_t M = (int64_t)(prefix + run);
    J.count[0] = M;
    if (M > J.tcap) flag_status(J.count, gs::kStatusCapacity);
  }
  for (int64_t c = c_begin; c < c_end; ++c) {
    uint32_t cnt[kPer];
    uint4 rec[kPer];
    uint32_t sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t i = c * kScanChunk + tid * kPer + j;
      rec[j] = i < n ? J.grec[i] : make_uint4(0u, 0u, 0u, 0u);  // this thread's own S1 writes
      cnt[j] = (rec[j].z & 0xffffu) * (rec[j].z >> 16);
      sum += cnt[j];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    __syncthreads();
    if (lane == 31) S.wsum[warp] = incl;
    __syncthreads();
    uint32_t woff = 0, total = 0;
    for (int w = 0; w < kSortWarps; ++w) {
      const uint32_t x = S.wsum[w];
      if (w < warp) woff += x;
      total += x;
    }
    int64_t go = (int64_t)prefix + woff + incl - sum;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t i = c * kScanChunk + tid * kPer + j;
      if (i < n) {
        rec[j].x = (uint32_t)min(go, (int64_t)0xFFFFFFFF);
        J.grec[i] = rec[j];
        for (int64_t sb = (go + kSlice - 1) / kSlice * kSlice; sb < go + cnt[j] && sb < J.tcap; sb += kSlice)
          J.slice_first[sb / kSlice] = (uint32_t)i;
      }
      go += cnt[j];
    }
    prefix += total;
  }
  return true;
}

// Stable ranks of a warp's ITEMS x 32 keys by digit (key >> shift) & 255 within the warp, in
// item-major order: peer masks of all items first, then the per-warp counts in item order
// (rank[] holds the peer mask until it is replaced by the rank).  Peers: every lane ORs its
// bit into its digit's word of a per-warp shared-memory table, reads the word back and clears
// it.  kFull: every item takes part (a full radix tile: no masks, no divergence); otherwise
// bit i of vbits says whether item i does.  Leaves the warp's digit counts in S.whist[warp].
template <int ITEMS, bool kFull>
__device__ __forceinline__ void rank_items(SortSmem<ITEMS>& S, const uint32_t (&k)[ITEMS], uint32_t vbits, int shift,
                                           uint32_t (&rank)[ITEMS]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const bool valid = kFull || ((vbits >> i) & 1u);
    const uint32_t d = (k[i] >> shift) & 255u;
    if (valid) atomicOr(&S.peer[warp][d], 1u << lane);
    __syncwarp();
    rank[i] = valid ? S.peer[warp][d] : 0u;
    __syncwarp();
    if (valid) S.peer[warp][d] = 0u;
    __syncwarp();
  }
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const uint32_t d = (k[i] >> shift) & 255u;
    const uint32_t peers = rank[i];
    // every peer stores the same new count (one of the identical stores lands)
    if (kFull) {
      const uint32_t before = S.whist[warp][d];
      __syncwarp();
      S.whist[warp][d] = before + __popc(peers);
      __syncwarp();
      rank[i] = before + __popc(peers & lt_mask);
    } else {
      const bool valid = (vbits >> i) & 1u;
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t before = S.whist[warp][d];
        __syncwarp(vmask);
        S.whist[warp][d] = before + __popc(peers);
        __syncwarp(vmask);
        rank[i] = before + __popc(peers & lt_mask);
      }
    }
  }
}

// All passes of one sort, run by the G CTAs bid = 0 .. G-1 that the job owns.
template <int ITEMS, bool kTileSort>
__device__ __forceinline__ void radix_body(const RadixJob& J, const uint32_t G, const uint32_t bid) {
  constexpr int kTile = kSortThreads * ITEMS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SortSmem<ITEMS>& S = *reinterpret_cast<SortSmem<ITEMS>*>(smem_raw);
  if (J.count[1] != 0) return;
  int64_t M = J.n_host >= 0 ? J.n_host : min(J.count[0], J.cap);  // keys of the pass (depth: visible after pass 0)
  int64_t ntiles = sort_tiles<ITEMS>(M);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kSortWarps * 256; i += kSortThreads) (&S.peer[0][0])[i] = 0u;
  uint32_t nbar = 0;
  for (int p = 0; p < J.passes; ++p) {
    const int shift = 8 * p;
    const bool gen = kTileSort && p == 0;
    const bool fin = kTileSort && p == J.passes - 1;
    const bool compact = !kTileSort && p == 0;  // drops the culled keys
    const uint32_t* kin = J.key[p & 1];
    const uint32_t* vin = J.val[p & 1];
    // ---- A: digit counts of every radix tile
    if (!kTileSort && p == 0) depth_phase0(S, J, J.n_host, ntiles, G, bid);
    if (gen) {
      for (int64_t tile = bid; tile < ntiles; tile += G) {
        for (int i = tid; i < 256; i += kSortThreads) S.tstart[i] = 0u;
        __syncthreads();
        const int64_t base = tile * kTile;
        gen_digit_counts(S, J, tile, base, (int)min((int64_t)kTile, M - base), M);
        J.hist[(int64_t)tid * J.hist_stride + tile] = S.tstart[tid];
        __syncthreads();
      }
    } else if (kTileSort || p > 0) {
      // the counts need the keys only; the next radix tile's keys are in flight while this
      // one's are counted
      uint32_t k[ITEMS];
      load_words<ITEMS>(kin, bid, M, k);
      for (int64_t tile = bid; tile < ntiles; tile += G) {
        for (int i = tid; i < 256; i += kSortThreads) S.tstart[i] = 0u;
        __syncthreads();
        const int nvalid = (int)min((int64_t)kTile, M - tile * kTile);
        uint32_t kn[ITEMS];
        load_words<ITEMS>(kin, tile + G, M, kn);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
          const int li = warp * (ITEMS * 32) + i * 32 + lane;
          if (li < nvalid) atomicAdd(&S.tstart[(k[i] >> shift) & 255u], 1u);
        }
        __syncthreads();
        J.hist[(int64_t)tid * J.hist_stride + tile] = S.tstart[tid];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) k[i] = kn[i];
      }
    }
    ++nbar;
    if (!grid_barrier(S, J, nbar * G, !(J.drop_arrival && nbar == 1 && bid == 0))) return;
    // ---- B: per digit, exclusive scan of its counts over the tiles; the column's sum is the
    // digit's total, from which phase C takes the digit bases
    // (twelve counts per thread as three 16-byte loads, the next twelve in flight while these
    // are scanned; counts past the last tile read as 0, and the row padding takes junk)
    for (uint32_t d = bid; d < 256; d += G) {
      uint32_t* col = J.hist + (int64_t)d * J.hist_stride;
      uint32_t carry = 0;
      constexpr int kPer = 12;
      constexpr int64_t kStep = kSortThreads * kPer;
      auto load = [&](int64_t c0, uint32_t (&y)[kPer]) {
#pragma unroll
        for (int q = 0; q < kPer / 4; ++q) {
          const int64_t t = c0 + tid * kPer + 4 * q;
          const uint4 v4 = t < ntiles ? __ldcg(reinterpret_cast<const uint4*>(col + t)) : make_uint4(0u, 0u, 0u, 0u);
          y[4 * q] = v4.x;
          y[4 * q + 1] = t + 1 < ntiles ? v4.y : 0u;
          y[4 * q + 2] = t + 2 < ntiles ? v4.z : 0u;
          y[4 * q + 3] = t + 3 < ntiles ? v4.w : 0u;
        }
      };
      uint32_t x[kPer];
      load(0, x);
      for (int64_t c0 = 0; c0 < ntiles; c0 += kStep) {
        uint32_t xn[kPer];
        load(c0 + kStep, xn);
        uint32_t sum = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) sum += x[j];
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane == 31) S.wsum[warp] = incl;
        __syncthreads();
        uint32_t run = carry + incl - sum, total = 0;
        for (int w = 0; w < kSortWarps; ++w) {
          const uint32_t s = S.wsum[w];
          if (w < warp) run += s;
          total += s;
        }
        uint32_t out[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          out[j] = run;
          run += x[j];
        }
#pragma unroll
        for (int q = 0; q < kPer / 4; ++q) {
          const int64_t t = c0 + tid * kPer + 4 * q;
          if (t < ntiles)
            *reinterpret_cast<uint4*>(col + t) = make_uint4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
        }
        carry += total;
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kPer; ++j) x[j] = xn[j];
      }
      if (tid == 0) J.small[kSmHist + (J.slot0 + p) * 256 + d] = carry;
    }
    if (!grid_barrier(S, J, ++nbar * G, true)) return;
    {  // the digit bases: exclusive scan of the digit totals (thread = digit)
      const uint32_t c = __ldcg(&J.small[kSmHist + (J.slot0 + p) * 256 + tid]);
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) S.wsum[warp] = incl;
      __syncthreads();
      uint32_t woff = 0;
      for (int w = 0; w < warp; ++w) woff += S.wsum[w];
      S.dbase[tid] = woff + incl - c;
      if (tid == 255) {
        S.total = woff + incl;
        if (compact && bid == 0) J.small[kSmVisible] = woff + incl;
      }
      __syncthreads();
    }
    // ---- C: rank within the tile, scatter through shared memory, digit-contiguous writes
    // The CTAs take radix tiles from a shared counter (the next one fetched while this one is
    // processed), so a CTA whose tiles were cheaper takes more: the phase ends when the work
    // does, not when the slowest CTA's fixed share does.  Thread 0 writes nxt[cur ^ 1] while
    // every thread reads nxt[cur]; each iteration ends with a block barrier.
    uint32_t* kout = J.key[(p + 1) & 1];
    uint32_t* vout = fin ? J.vals_out : J.val[(p + 1) & 1];
    const int ctr = kSmTileCtr + J.sort_id * kMaxTilePasses + p;
    if (tid == 0) S.nxt[0] = atomicAdd(&J.small[ctr], 1u);
    __syncthreads();
    uint32_t cur = 0;
    for (uint32_t tile = S.nxt[0]; tile < ntiles; cur ^= 1u, tile = S.nxt[cur]) {
      if (tid == 0) S.nxt[cur ^ 1u] = atomicAdd(&J.small[ctr], 1u);
      // this tile's global digit offsets, loaded now and used after the ranking
      const uint32_t tile_base = S.dbase[tid] + __ldcg(&J.hist[(int64_t)tid * J.hist_stride + tile]);
      const int64_t base = tile * kTile;
      const int nvalid = (int)min((int64_t)kTile, M - base);
      const bool full = nvalid == kTile && !compact;
      // (loading the next tile's keys during this one's write-out was measured slower: the
      // extra live registers spill)
      uint32_t k[ITEMS], v[ITEMS], rank[ITEMS];
      if (gen) {
        gen_tile<ITEMS>(S, J, tile, base, nvalid, k, v);
      } else {
        load_words<ITEMS>(kin, tile, M, k);
        load_words<ITEMS>(vin, tile, M, v);
      }
      for (int i = tid; i < kSortWarps * 256; i += kSortThreads) (&S.whist[0][0])[i] = 0u;
      __syncthreads();
      const int wbase = warp * (ITEMS * 32);
      uint32_t vbits = 0;  // bit i: item i takes part (in range; in pass 0 of the depth sort, visible)
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const int li = wbase + i * 32 + lane;
        if (full || (li < nvalid && !(compact && k[i] == kCulledKey))) vbits |= 1u << i;
      }
      if (full) rank_items<ITEMS, true>(S, k, 0u, shift, rank);
      else rank_items<ITEMS, false>(S, k, vbits, shift, rank);
      __syncthreads();
      {  // per digit (thread = digit): the tile's offsets.  S.whist[w][d] becomes warp w's first
         // staging slot for digit d, S.gbase[d] the output slot of staging slot 0 (mod 2^32)
        const int d = tid;
        uint32_t run = 0;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) run += S.whist[w][d];
        const uint32_t cnt = run;
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
        const uint32_t ts = woff + incl - cnt;  // the digit's first staging slot
        uint32_t r = ts;
#pragma unroll
        for (int w = 0; w < kSortWarps; ++w) {
          const uint32_t c = S.whist[w][d];
          S.whist[w][d] = r;
          r += c;
        }
        S.gbase[d] = tile_base - ts;
        if (d == 255) S.tvalid = woff + incl;
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        if ((vbits >> i) & 1u) {
          const uint32_t d = (k[i] >> shift) & 255u;
          const uint32_t pos = S.whist[warp][d] + rank[i];
          S.keys[pos] = k[i];
          S.vals[pos] = v[i];
        }
      }
      __syncthreads();

#pragma unroll 4
      for (int i = 0; i < ITEMS; ++i) {
        const int q = i * kSortThreads + tid;
        if (q < (int)S.tvalid) {
          const uint32_t key = S.keys[q];
          const uint32_t d = (key >> shift) & 255u;
          const uint32_t g = S.gbase[d] + (uint32_t)q;
          if (g < (uint64_t)M) {  // always true unless a barrier gave up (status bit set)
            const uint32_t val = S.vals[q];
            kout[g] = key;  // the last tile pass keeps the sorted tile ids for the ranges
            if (fin && J.keys64) J.keys64[g] = ((uint64_t)key << 32) | __float_as_uint(__ldg(&J.q0[val].z));
            vout[g] = val;
          }
        }
      }
      __syncthreads();
    }
    if (compact) {  // the later passes sort the visible keys, written to [0, total) by this one
      M = S.total;
      ntiles = sort_tiles<ITEMS>(M);
    }
    if (p + 1 < J.passes && !grid_barrier(S, J, ++nbar * G, true)) return;
  }
  if (!grid_barrier(S, J, ++nbar * G, true)) return;
  if (!kTileSort) {
    depth_scan(S, J, M, G, bid, nbar);
  } else {
    // the staged ranges: tile t's run of sorted instances starts where the tile id changes
    // (the host zeroed them, so empty tiles keep [0, 0)).  Four sorted ids per thread in one
    // 16-byte load (the buffer is 256-byte aligned and its padding covers the last group), four
    // such groups per round; a thread's neighbours come from the lanes beside it, a warp's
    // edges from one more load.
    const uint32_t* skey = J.key[J.passes & 1];
    const uint4* sk4 = reinterpret_cast<const uint4*>(skey);
    const int64_t n4 = (M + 3) / 4;
    const int64_t span = (n4 + 31) / 32 * 32;  // whole warps, so the shuffles see every lane
    const int64_t stride = (int64_t)G * kSortThreads;
    constexpr int kU = 4;  // groups per thread per round, all of their loads in flight together
    for (int64_t q0 = (int64_t)bid * kSortThreads + tid; q0 < span; q0 += kU * stride) {
      uint4 v4[kU];
      uint32_t edge[kU];  // lane 0: the id before its group; lane 31: the id after
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t q = q0 + u * stride;
        const bool in = q < n4;
        v4[u] = in ? __ldcg(&sk4[q]) : make_uint4(0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu);
        edge[u] = 0xFFFFFFFFu;
        if (lane == 0 && in && q > 0) edge[u] = __ldcg(&skey[4 * q - 1]);
        if (lane == 31 && in && 4 * q + 4 < M) edge[u] = __ldcg(&skey[4 * q + 4]);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int64_t q = q0 + u * stride;
        if (q >= span) break;  // the same for the whole warp: span and stride are whole warps
        const bool in = q < n4;
        uint32_t e[6];
        e[0] = __shfl_up_sync(0xffffffffu, v4[u].w, 1);
        e[5] = __shfl_down_sync(0xffffffffu, v4[u].x, 1);
        if (lane == 0) e[0] = edge[u];
        if (lane == 31) e[5] = edge[u];
        e[1] = v4[u].x; e[2] = v4[u].y; e[3] = v4[u].z; e[4] = v4[u].w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int64_t g = 4 * q + j;
          if (!in || g >= M) break;
          const uint32_t t = e[j + 1];
          if (g == 0 || e[j] != t) J.rstage[2 * (int64_t)t] = (uint32_t)g;
          if (g == M - 1 || e[j + 2] != t) J.rstage[2 * (int64_t)t + 1] = (uint32_t)(g + 1);
        }
      }
    }
  }
}

// The sorts of up to kMaxSortViews views in one launch: CTAs [v G, (v + 1) G) sort view v,
// with their own barrier counter and workspace, so the views' barrier waits and uneven phases
// overlap.  A CTA reads its view's job in place, from kernel parameter space.
__global__ void __launch_bounds__(kSortThreads, 4) k_depth_sort(const __grid_constant__ RadixBatch B) {
  const uint32_t G = gridDim.x / (uint32_t)B.views;
  const uint32_t view = blockIdx.x / G;
  radix_body<kDepthItems, false>(B.job[view], G, blockIdx.x - view * G);
}

// The same with radix tiles of kTileItems keys, for large N: fewer tiles, so fewer digit
// counts to scan and less fixed work per key.
__global__ void __launch_bounds__(kSortThreads, GS_SORT_MIN_BLOCKS) k_depth_sort_wide(const __grid_constant__ RadixBatch B) {
  const uint32_t G = gridDim.x / (uint32_t)B.views;
  const uint32_t view = blockIdx.x / G;
  radix_body<kTileItems, false>(B.job[view], G, blockIdx.x - view * G);
}

#ifndef GS_TILE_MIN_BLOCKS
#define GS_TILE_MIN_BLOCKS GS_SORT_MIN_BLOCKS
#endif
__global__ void __launch_bounds__(kSortThreads, GS_TILE_MIN_BLOCKS) k_tile_sort(const __grid_constant__ RadixBatch B) {
  const uint32_t G = gridDim.x / (uint32_t)B.views;
  const uint32_t view = blockIdx.x / G;
  radix_body<kTileItems, true>(B.job[view], G, blockIdx.x - view * G);
}

// Per view of a batch: the buffers zeroed before the sorts (the status words, the small
// block, the difference grid, the caller's ranges) and the staged ranges published after.
struct ViewBuffers {
  uint32_t* zero[kMaxSortViews][4];
  int64_t zero_words[kMaxSortViews][4];
  const uint32_t* rstage[kMaxSortViews];
  uint32_t* ranges[kMaxSortViews];
  const int64_t* count[kMaxSortViews];
  int64_t words2T[kMaxSortViews];  // 2 x tiles of the view
  int views;
};

// blockIdx.y = view * 4 + buffer
__global__ void k_sort_init(const __grid_constant__ ViewBuffers B) {
  const int v = blockIdx.y >> 2, b = blockIdx.y & 3;
  uint32_t* p = B.zero[v][b];
  const int64_t words = B.zero_words[v][b];
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0u;
}

// Copies every view's staged tile ranges to the caller once all its passes finished cleanly
// (blockIdx.y = view).
__global__ void k_publish_ranges(const __grid_constant__ ViewBuffers B) {
  const int v = blockIdx.y;
  if (B.count[v][1] != 0) return;
  const uint32_t* src = B.rstage[v];
  uint32_t* dst = B.ranges[v];
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < B.words2T[v]; i += stride) dst[i] = src[i];
}

// Resident CTAs per SM of a sort kernel for a given dynamic shared-memory size on the current
// device (the shared-memory attribute and the occupancy answer are both kept per device).
template <int kKernel>  // 0: depth sort, 1: tile sort, 2: depth sort with wide radix tiles
int radix_blocks_per_sm(size_t smem) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static size_t cached_smem[kMaxDev] = {0};
  static int cached[kMaxDev] = {0};
  const void* fn = kKernel == 1 ? (const void*)k_tile_sort
                                : (kKernel == 2 ? (const void*)k_depth_sort_wide : (const void*)k_depth_sort);
  gs::max_dynamic_smem(fn, (int)smem);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = -1;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && cached[dev] > 0 && cached_smem[dev] == smem) return cached[dev];
  int b = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, kSortThreads, smem) != cudaSuccess || b < 1) b = 1;
  if (dev >= 0) {
    cached[dev] = b;
    cached_smem[dev] = smem;
  }
  return b;
}

// Cooperative launches: every CTA of the grid is resident at once, which the grid barriers need.
cudaError_t launch_tile_sort(const RadixBatch& batch, int grid, size_t smem, cudaStream_t st) {
  RadixBatch b = batch;
  void* args[] = {&b};
  return cudaLaunchCooperativeKernel((const void*)k_tile_sort, dim3(grid), dim3(kSortThreads), args, smem, st);
}
cudaError_t launch_depth_sort(const RadixBatch& batch, int grid, size_t smem, cudaStream_t st, bool wide) {
  RadixBatch b = batch;
  void* args[] = {&b};
  return cudaLaunchCooperativeKernel(wide ? (const void*)k_depth_sort_wide : (const void*)k_depth_sort, dim3(grid),
                                     dim3(kSortThreads), args, smem, st);
}


// Views per tile-sort launch for a capacity (see kTileBudgetBytes).
int tile_group(int views, int64_t cap) {
  const double per_view = 16.0 * (double)std::max<int64_t>(cap, 1) + 1024.0 * (double)sort_tiles<kTileItems>(cap);
  const int fit = (int)std::min<double>(kMaxSortViews, std::floor(kTileBudgetBytes / per_view));
  return std::max(1, std::min({fit, views, kMaxSortViews}));
}

// Largest tile count over a batch of cameras.
int64_t batch_tiles(const gs::Cam* k, int views) {
  int64_t T = 1;
  for (int v = 0; v < views; ++v) T = std::max(T, (int64_t)k[v].Tx * k[v].Ty);
  return T;
}

struct SortView {
  const float* proj;
  gs::Cam k;
  uint64_t* keys;
  uint32_t* vals;
  uint32_t* ranges;
  int64_t* count;
};

// Enqueues the sorts of `views` views that share n and capacity.  Views go in groups of up
// to kMaxSortViews: one zeroing launch, one depth-sort launch, one tile sort per view, one
// publishing launch.  A group's depth buffers are w[0 .. group size), reused by the next group
// once the tile sorts before it (which read them) are enqueued.
gs_status run_sorts(const SortView* V, int views, int64_t n, int64_t capacity, const Workspace* w, int tg,
                    cudaStream_t st) {
  const int64_t limit = gs::wait_limit();
  const int drop = gs::take_drop_publish();
  const int sms = gs::num_sms();
  for (int g0 = 0; g0 < views; g0 += kMaxSortViews) {
    const int gv = std::min(kMaxSortViews, views - g0);
    ViewBuffers vb{};
    vb.views = gv;
    int64_t max_words = 0;
    for (int v = 0; v < gv; ++v) {
      const gs::Cam& k = V[g0 + v].k;
      const int64_t T = (int64_t)k.Tx * k.Ty;
      uint32_t* z[4] = {reinterpret_cast<uint32_t*>(V[g0 + v].count), w[v].small, w[v].rstage, V[g0 + v].ranges};
      const int64_t zw[4] = {4, kSmWords, 2 * T, 2 * T};
      for (int b = 0; b < 4; ++b) {
        vb.zero[v][b] = z[b];
        vb.zero_words[v][b] = zw[b];
        max_words = std::max(max_words, zw[b]);
      }
      vb.rstage[v] = w[v].rstage;
      vb.ranges[v] = V[g0 + v].ranges;
      vb.count[v] = V[g0 + v].count;
      vb.words2T[v] = 2 * T;
    }
    const int zx = (int)std::min<int64_t>(std::max<int64_t>(1, (max_words + 1023) / 1024), 64);
    k_sort_init<<<dim3(zx, 4 * gv), 256, 0, st>>>(vb);
    if (gs_status s = gs::check_launch("gs_bin_sort init")) return s;
    if (n == 0) continue;
    // 1. per view, Gaussians by (depth, index): 4 stable passes over 32-bit depth keys; phase
    //    0 also writes every Gaussian's tile-rectangle record, and after the passes the
    //    tiles-touched scan gives every sorted Gaussian's first slot (and M)
    RadixBatch db{};
    db.views = gv;
    const bool wide = n >= kWideDepthN;
    const size_t dsmem = wide ? sizeof(SortSmem<kTileItems>) : sizeof(SortSmem<kDepthItems>);
    const int64_t dtiles = wide ? sort_tiles<kTileItems>(n) : sort_tiles<kDepthItems>(n);
    for (int v = 0; v < gv; ++v) {
      const SortView& sv = V[g0 + v];
      RadixJob& dj = db.job[v];
      dj.key[0] = w[v].dkey[0]; dj.key[1] = w[v].dkey[1];
      dj.val[0] = w[v].didx[0]; dj.val[1] = w[v].didx[1];
      dj.n_host = n; dj.cap = n; dj.passes = kDepthPasses; dj.slot0 = 0; dj.sort_id = 0;
      dj.hist = w[v].hist_depth; dj.hist_stride = hist_cols(dtiles);
      dj.small = w[v].small; dj.count = sv.count; dj.limit = limit; dj.drop_arrival = drop == 2 && g0 + v == 0;
      dj.proj = sv.proj; dj.Tx = sv.k.Tx; dj.Ty = sv.k.Ty; dj.rrec = w[v].rrec;
      dj.cta_tot = w[v].cta_tot; dj.grec = w[v].grec; dj.slice_first = w[v].slice_first; dj.tcap = capacity;
    }
    // CTAs per view: as many as the radix tiles if the group fits, else an equal share of the
    // resident CTAs
    const int64_t resident = (int64_t)sms * (wide ? radix_blocks_per_sm<2>(dsmem) : radix_blocks_per_sm<0>(dsmem));
    const int64_t G = std::max<int64_t>(1, std::min<int64_t>({std::max<int64_t>(dtiles, kMinSortCtas), resident / gv,
                                                              (int64_t)kMaxScanCtas}));
    if (cudaError_t e = launch_depth_sort(db, (int)(G * gv), dsmem, st, wide))
      return gs::set_error(GS_ERR_CUDA, "gs_bin_sort depth sort: %s", cudaGetErrorString(e));
    if (gs_status s = gs::check_launch("gs_bin_sort depth sort")) return s;
    // 2. per view, the stable sort of the instances by tile id: the first pass generates the
    //    (tile, index) pairs in depth order from the scan's records, the last writes the
    //    caller's arrays; tg views per launch, each with its own ping-pong buffers
    const size_t tsmem = sizeof(SortSmem<kTileItems>);
    const int64_t tresident = (int64_t)sms * radix_blocks_per_sm<1>(tsmem);
    for (int t0 = 0; t0 < gv; t0 += tg) {
      const int tv = std::min(tg, gv - t0);
      RadixBatch tb{};
      tb.views = tv;
      for (int j = 0; j < tv; ++j) {
        const int v = t0 + j;
        const SortView& sv = V[g0 + v];
        RadixJob& tj = tb.job[j];
        tj.key[0] = w[v].tkey[0]; tj.key[1] = w[v].tkey[1];
        tj.val[0] = w[v].tval[0]; tj.val[1] = w[v].tval[1];
        tj.n_host = -1; tj.cap = capacity; tj.passes = tile_passes(sv.k);
        tj.slot0 = kDepthPasses; tj.sort_id = 1;
        tj.hist = w[v].hist_tile; tj.hist_stride = hist_cols(sort_tiles<kTileItems>(capacity));
        tj.small = w[v].small; tj.count = sv.count; tj.limit = limit; tj.drop_arrival = drop == 1 && g0 + v == 0;
        tj.gen = GenSource{w[v].slice_first, w[v].grec, sv.k.Tx};
        tj.q0 = reinterpret_cast<const float4*>(sv.proj); tj.keys64 = sv.keys; tj.vals_out = sv.vals;
        tj.rstage = w[v].rstage;
      }
      const int64_t TG =
          std::max<int64_t>(1, std::min<int64_t>(tresident / tv, std::max<int64_t>(sort_tiles<kTileItems>(capacity), kMinSortCtas)));
      if (cudaError_t e = launch_tile_sort(tb, (int)(TG * tv), tsmem, st))
        return gs::set_error(GS_ERR_CUDA, "gs_bin_sort tile sort: %s", cudaGetErrorString(e));
      if (gs_status s = gs::check_launch("gs_bin_sort tile sort")) return s;
    }
    k_publish_ranges<<<dim3(sms, gv), 256, 0, st>>>(vb);
    if (gs_status s = gs::check_launch("gs_bin_sort ranges")) return s;
  }
  return GS_OK;
}

// Reads back the status words of `views` views (count[2v], count[2v + 1]) after a sort.
gs_status read_counts(const int64_t* const* count, int views, int64_t* count_host, cudaStream_t st) {
  std::vector<int64_t> hc(2 * (size_t)views, 0);
  for (int v = 0; v < views; ++v)
    if (cudaMemcpyAsync(&hc[2 * v], count[v], 2 * sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
      return gs::check_launch("gs_bin_sort count readback");
  if (cudaStreamSynchronize(st) != cudaSuccess) return gs::check_launch("gs_bin_sort count readback");
  int64_t bits = 0;
  for (int v = 0; v < views; ++v) {
    count_host[v] = hc[2 * v];
    bits |= hc[2 * v + 1];
  }
  if (bits & gs::kStatusTimeout) return gs::set_error(GS_ERR_TIMEOUT, "gs_bin_sort: a bounded device-side wait gave up");
  if (bits & gs::kStatusCapacity) {
    int64_t worst = 0;
    for (int v = 0; v < views; ++v) worst = std::max(worst, count_host[v]);
    return gs::set_error(GS_ERR_CAPACITY, "gs_bin_sort: %lld instances exceed the capacity", (long long)worst);
  }
  return GS_OK;
}

gs_status check_sort_args(int64_t n, int64_t capacity, const gs::Cam& k, const char* fn) {
  if (n < 0 || n >= (int64_t(1) << 31)) return gs::set_error(GS_ERR_INVALID, "%s: bad n", fn);
  if (capacity < 0 || capacity >= (int64_t(1) << 30))
    return gs::set_error(GS_ERR_INVALID, "%s: capacity must be in [0, 2^30)", fn);
  if (tile_passes(k) > kMaxTilePasses || k.Tx > 65535 || k.Ty > 65535)  // 16-bit rectangle fields
    return gs::set_error(GS_ERR_INVALID, "%s: %d x %d tiles exceed the supported grid", fn, k.Tx, k.Ty);
  return GS_OK;
}

}  // namespace

extern "C" size_t gs_bin_sort_workspace_size(int64_t n, int64_t capacity, const gs_camera* cam) {
  return gs_bin_sort_batch_workspace_size(1, n, capacity, cam);
}

extern "C" size_t gs_bin_sort_batch_workspace_size(int batch, int64_t n, int64_t capacity, const gs_camera* cams) {
  if (!cams || batch < 1 || n < 0 || capacity < 0) return 0;
  std::vector<gs::Cam> k((size_t)batch);
  for (int v = 0; v < batch; ++v) k[v] = gs::make_cam(cams[v]);
  return carve(nullptr, nullptr, std::min(batch, kMaxSortViews), n, capacity, batch_tiles(k.data(), batch),
               tile_group(batch, capacity));
}

extern "C" gs_status gs_bin_sort(const float* proj, int64_t n, const gs_camera* cam, void* workspace,
                                 size_t workspace_bytes, uint64_t* keys, uint32_t* vals, int64_t capacity,
                                 uint32_t* ranges, int64_t* count, int64_t* count_host, void* stream) {
  if (gs_status s = gs::check_camera(cam)) return s;
  const gs::Cam k = gs::make_cam(*cam);
  if (gs_status s = check_sort_args(n, capacity, k, "gs_bin_sort")) return s;
  if (!count || !ranges || (n > 0 && !proj) || (capacity > 0 && !vals) || !workspace)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: NULL pointer");
  if ((proj && !gs::aligned16(proj)) || !gs::aligned8(count) || (keys && !gs::aligned8(keys)) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: misaligned pointer");
  const size_t need = gs_bin_sort_workspace_size(n, capacity, cam);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort: workspace %zu bytes < %zu needed", workspace_bytes, need);
  Workspace w;
  carve(&w, reinterpret_cast<char*>(workspace), 1, n, capacity, (int64_t)k.Tx * k.Ty, 1);
  cudaStream_t st = gs::as_stream(stream);
  const SortView view{proj, k, keys, vals, ranges, count};
  if (gs_status s = run_sorts(&view, 1, n, capacity, &w, 1, st)) return s;
  if (!count_host) return GS_OK;
  const int64_t* c = count;
  return read_counts(&c, 1, count_host, st);
}

extern "C" gs_status gs_bin_sort_batch(const float* const* projs, int batch, int64_t n, const gs_camera* cams,
                                       void* workspace, size_t workspace_bytes, uint64_t* const* keys,
                                       uint32_t* const* vals, int64_t capacity, uint32_t* const* ranges,
                                       int64_t* counts, int64_t* counts_host, void* stream) {
  if (batch < 1) return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: batch must be >= 1");
  if (!projs || !cams || !vals || !ranges || !counts || !workspace)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: NULL pointer");
  std::vector<SortView> V((size_t)batch);
  for (int v = 0; v < batch; ++v) {
    if (gs_status s = gs::check_camera(&cams[v])) return s;
    SortView& sv = V[v];
    sv = SortView{projs[v], gs::make_cam(cams[v]), keys ? keys[v] : nullptr, vals[v], ranges[v], counts + 2 * v};
    if (gs_status s = check_sort_args(n, capacity, sv.k, "gs_bin_sort_batch")) return s;
    if (!sv.ranges || (n > 0 && !sv.proj) || (capacity > 0 && !sv.vals))
      return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: NULL pointer (view %d)", v);
    if ((sv.proj && !gs::aligned16(sv.proj)) || (sv.keys && !gs::aligned8(sv.keys)))
      return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: misaligned pointer (view %d)", v);
  }
  if (!gs::aligned8(counts) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: misaligned pointer");
  const size_t need = gs_bin_sort_batch_workspace_size(batch, n, capacity, cams);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_bin_sort_batch: workspace %zu bytes < %zu needed", workspace_bytes,
                         need);
  std::vector<gs::Cam> k((size_t)batch);
  for (int v = 0; v < batch; ++v) k[v] = V[v].k;
  Workspace w[kMaxSortViews];
  carve(w, reinterpret_cast<char*>(workspace), std::min(batch, kMaxSortViews), n, capacity,
        batch_tiles(k.data(), batch), tile_group(batch, capacity));
  cudaStream_t st = gs::as_stream(stream);
  if (gs_status s = run_sorts(V.data(), batch, n, capacity, w, tile_group(batch, capacity), st)) return s;
  if (!counts_host) return GS_OK;
  std::vector<const int64_t*> c((size_t)batch);
  for (int v = 0; v < batch; ++v) c[v] = counts + 2 * v;
  return read_counts(c.data(), batch, counts_host, st);
}
