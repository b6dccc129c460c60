// Opacity pruning (gs_prune): the pruning half of the densification step of the Grendel-GS
// training flow (训练流程: "prune low-opacity Gaussians").  Gaussian i is kept when its
// opacity logit (plane 0, w) is at least min_logit -- sigmoid is increasing, so this is
// opacity >= sigmoid(min_logit) -- and its planes in every set (parameters, Adam moments)
// move to the next free slot, index order preserved.  A stable stream compaction:
//   k_prune_count    per 256-Gaussian block, the number kept;
//   k_prune_scan     one CTA: exclusive scan of the block counts, the total to n_keep;
//   k_prune_scatter  per block, each kept Gaussian's rank (warp ballots, warp offsets) and
//                    the copy of its 15 float4 planes of every set (coalesced plane by plane).
#include "common.cuh"

namespace {

constexpr int kPruneThreads = 256;
constexpr int kPruneScan = 1024;
constexpr int kMaxSets = 4;

struct PruneSets {
  const float4* in[kMaxSets];
  float4* out[kMaxSets];
  int n_sets;
};

__device__ __forceinline__ bool kept(const float4* __restrict__ p0, int64_t i, float min_logit) {
  return __ldg(&p0[i].w) >= min_logit;  // false for a NaN logit
}

__global__ void __launch_bounds__(kPruneThreads) k_prune_count(const float4* __restrict__ p0, int64_t n, float min_logit,
                                                               uint32_t* __restrict__ counts) {
  __shared__ uint32_t s_w[kPruneThreads / 32];
  const int64_t i = (int64_t)blockIdx.x * kPruneThreads + threadIdx.x;
  const bool k = i < n && kept(p0, i, min_logit);
  const uint32_t b = __ballot_sync(0xffffffffu, k);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = __popc(b);
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t s = 0;
    for (int w = 0; w < kPruneThreads / 32; ++w) s += s_w[w];
    counts[blockIdx.x] = s;
  }
}

__global__ void __launch_bounds__(kPruneScan) k_prune_scan(const uint32_t* __restrict__ counts, int64_t nb,
                                                           int64_t* __restrict__ offsets, int64_t* __restrict__ n_keep) {
  __shared__ long long s_warp[kPruneScan / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (nb + kPruneScan - 1) / kPruneScan;
  const int64_t b0 = min(nb, (int64_t)tid * per), b1 = min(nb, b0 + per);
  long long sum = 0;
  for (int64_t b = b0; b < b1; ++b) sum += counts[b];
  long long incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int w = 0; w < kPruneScan / 32; ++w) {
      const long long c = s_warp[w];
      s_warp[w] = run;
      run += c;
    }
    *n_keep = run;
  }
  __syncthreads();
  long long run = s_warp[warp] + incl - sum;
  for (int64_t b = b0; b < b1; ++b) {
    offsets[b] = run;
    run += counts[b];
  }
}

__global__ void __launch_bounds__(kPruneThreads) k_prune_scatter(const __grid_constant__ PruneSets S, int64_t n,
                                                                 float min_logit, const int64_t* __restrict__ offsets,
                                                                 int64_t out_stride) {
  __shared__ uint32_t s_w[kPruneThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * kPruneThreads + threadIdx.x;
  const bool k = i < n && kept(S.in[0], i, min_logit);
  const uint32_t b = __ballot_sync(0xffffffffu, k);
  if (lane == 0) s_w[warp] = __popc(b);
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; ++w) before += s_w[w];
  if (!k) return;
  const int64_t dst = offsets[blockIdx.x] + before + __popc(b & ((1u << lane) - 1u));
  if (dst >= out_stride) return;  // more kept than the output holds: reported by the host
  for (int s = 0; s < S.n_sets; ++s) {
    const float4* src = S.in[s];
    float4* out = S.out[s];
#pragma unroll
    for (int pl = 0; pl < 15; ++pl) out[(int64_t)pl * out_stride + dst] = __ldg(&src[(int64_t)pl * n + i]);
  }
}

int64_t prune_blocks(int64_t n) { return (n + kPruneThreads - 1) / kPruneThreads; }

}  // namespace

extern "C" size_t gs_prune_workspace_size(int64_t n) {
  if (n < 0) return 0;
  const size_t nb = (size_t)prune_blocks(n);
  return ((sizeof(uint32_t) * nb + 255) & ~size_t(255)) + sizeof(int64_t) * nb;
}

extern "C" gs_status gs_prune(const float* const* planes_in, int n_sets, int64_t n, float min_logit,
                              float* const* planes_out, int64_t out_stride, void* workspace, size_t workspace_bytes,
                              int64_t* n_keep, int64_t* n_keep_host, void* stream) {
  if (n_sets < 1 || n_sets > kMaxSets) return gs::set_error(GS_ERR_INVALID, "gs_prune: n_sets must be 1..%d", kMaxSets);
  if (n < 0 || n > (int64_t(1) << 31) || out_stride < 0)
    return gs::set_error(GS_ERR_INVALID, "gs_prune: bad n or out_stride");
  if (!planes_in || !n_keep || (out_stride > 0 && !planes_out) || (n > 0 && !workspace))
    return gs::set_error(GS_ERR_INVALID, "gs_prune: NULL pointer");
  if (!gs::aligned8(n_keep) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_prune: misaligned pointer");
  PruneSets S{};
  S.n_sets = n_sets;
  for (int s = 0; s < n_sets; ++s) {
    if (n > 0 && (!planes_in[s] || !gs::aligned16(planes_in[s])))
      return gs::set_error(GS_ERR_INVALID, "gs_prune: input set %d NULL or misaligned", s);
    if (out_stride > 0 && (!planes_out[s] || !gs::aligned16(planes_out[s])))
      return gs::set_error(GS_ERR_INVALID, "gs_prune: output set %d NULL or misaligned", s);
    S.in[s] = reinterpret_cast<const float4*>(planes_in[s]);
    S.out[s] = out_stride > 0 ? reinterpret_cast<float4*>(planes_out[s]) : nullptr;
  }
  cudaStream_t st = gs::as_stream(stream);
  if (n == 0) {
    if (cudaMemsetAsync(n_keep, 0, sizeof(int64_t), st) != cudaSuccess) return gs::check_launch("gs_prune");
  } else {
    const size_t need = gs_prune_workspace_size(n);
    if (workspace_bytes < need)
      return gs::set_error(GS_ERR_INVALID, "gs_prune: workspace %zu bytes < %zu needed", workspace_bytes, need);
    const int64_t nb = prune_blocks(n);
    uint32_t* counts = reinterpret_cast<uint32_t*>(workspace);
    int64_t* offsets = reinterpret_cast<int64_t*>(reinterpret_cast<char*>(workspace) +
                                                  ((sizeof(uint32_t) * (size_t)nb + 255) & ~size_t(255)));
    k_prune_count<<<(unsigned)nb, kPruneThreads, 0, st>>>(S.in[0], n, min_logit, counts);
    if (gs_status s = gs::check_launch("gs_prune count")) return s;
    k_prune_scan<<<1, kPruneScan, 0, st>>>(counts, nb, offsets, n_keep);
    if (gs_status s = gs::check_launch("gs_prune scan")) return s;
    if (out_stride > 0) {
      k_prune_scatter<<<(unsigned)nb, kPruneThreads, 0, st>>>(S, n, min_logit, offsets, out_stride);
      if (gs_status s = gs::check_launch("gs_prune scatter")) return s;
    }
  }
  if (!n_keep_host) return GS_OK;
  if (cudaMemcpyAsync(n_keep_host, n_keep, sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return gs::check_launch("gs_prune readback");
  if (out_stride > 0 && *n_keep_host > out_stride)
    return gs::set_error(GS_ERR_CAPACITY, "gs_prune: %lld kept exceed the output stride %lld",
                         (long long)*n_keep_host, (long long)out_stride);
  return GS_OK;
}
