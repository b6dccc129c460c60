// Densification, clone / split (gs_densify): the growing half of the densification step of
// the Grendel-GS training flow (训练流程: "致密化", clone or split the Gaussians that need
// more detail).  The pages give no criterion; the readings:
//   * the statistic (accumulated by gs_project_bwd / gs_project_bwd_adam): per Gaussian, the
//     sum over the views that see it of the length of its screen-space mean gradient, and the
//     number of those views;
//   * selected: seen at least once and sum / count >= grad_threshold (fp32);
//   * split if the largest log-scale exceeds log_scale_threshold, else clone;
//   * output: the Gaussians not split, in index order, then for every selected Gaussian in
//     index order its new ones: a clone (an exact copy), or two split children with means
//     mu + R(q / |q|) (s * z_k), s = exp(log-scale), z_k the caller's standard normals, and
//     log-scales lowered by ln 1.6, the rest copied; new Gaussians get zero Adam moments.
// A stable two-stream compaction:
//   k_densify_count    per 256-Gaussian block: kept Gaussians and new ones;
//   k_densify_scan     one CTA: exclusive scans of both, the totals;
//   k_densify_scatter  per block, every Gaussian's slots (warp ballots and scans) and the
//                      copies of its 15 float4 planes of parameters and moments.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kScan = 1024;
constexpr float kLn16 = 0.470003629245735553650937031148f;  // ln 1.6

// 0: untouched, 1: cloned, 2: split.  Comparisons in the order and precision the statistic is
// defined in: (float) sum / count against the threshold, and the largest log-scale (the
// larger of two taken as std::max does) against its threshold.
__device__ __forceinline__ int kind_of(const float4* __restrict__ p1, const float2* __restrict__ stat, int64_t i,
                                       float grad_threshold, float log_scale_threshold) {
  const float2 s = stat[i];
  if (!(s.y > 0.f)) return 0;
  const float avg = s.x / s.y;
  if (!(avg >= grad_threshold)) return 0;
  const float4 ls = __ldg(&p1[i]);
  float m = ls.x < ls.y ? ls.y : ls.x;
  m = m < ls.z ? ls.z : m;
  return m > log_scale_threshold ? 2 : 1;
}

struct Sets {
  const float4* p;
  const float4* m;
  const float4* v;
  float4* po;
  float4* mo;
  float4* vo;
};

// Per block: (Gaussians kept, new Gaussians).
__global__ void __launch_bounds__(kThreads) k_densify_count(const float4* __restrict__ p, const float2* __restrict__ stat,
                                                            int64_t n, float thr, float lthr,
                                                            uint32_t* __restrict__ counts) {
  __shared__ uint32_t s_k[kThreads / 32], s_n[kThreads / 32];
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int kind = i < n ? kind_of(p + n, stat, i, thr, lthr) : -1;
  uint32_t keep = (kind == 0 || kind == 1) ? 1u : 0u, add = kind == 1 ? 1u : (kind == 2 ? 2u : 0u);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    keep += __shfl_xor_sync(0xffffffffu, keep, o);
    add += __shfl_xor_sync(0xffffffffu, add, o);
  }
  if ((threadIdx.x & 31) == 0) {
    s_k[threadIdx.x >> 5] = keep;
    s_n[threadIdx.x >> 5] = add;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0, b = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      a += s_k[w];
      b += s_n[w];
    }
    counts[2 * blockIdx.x] = a;
    counts[2 * blockIdx.x + 1] = b;
  }
}

// Exclusive scans of the kept and new counts over the blocks (one CTA); totals[0] = output
// count, [1] clones, [2] splits, [3] kept.
__global__ void __launch_bounds__(kScan) k_densify_scan(const uint32_t* __restrict__ counts, int64_t nb, int64_t n,
                                                        int64_t* __restrict__ offsets, int64_t* __restrict__ totals) {
  __shared__ long long s_warp[2][kScan / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (nb + kScan - 1) / kScan;
  const int64_t b0 = min(nb, (int64_t)tid * per), b1 = min(nb, b0 + per);
  long long sum[2] = {0, 0};
  for (int64_t b = b0; b < b1; ++b) {
    sum[0] += counts[2 * b];
    sum[1] += counts[2 * b + 1];
  }
  long long incl[2] = {sum[0], sum[1]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const long long u = __shfl_up_sync(0xffffffffu, incl[c], o);
      if (lane >= o) incl[c] += u;
    }
  if (lane == 31) {
    s_warp[0][warp] = incl[0];
    s_warp[1][warp] = incl[1];
  }
  __syncthreads();
  if (tid < 2) {
    long long run = 0;
    for (int w = 0; w < kScan / 32; ++w) {
      const long long c = s_warp[tid][w];
      s_warp[tid][w] = run;
      run += c;
    }
    if (tid == 0) totals[3] = run;
    else totals[4] = run;
  }
  __syncthreads();
  if (tid == 0) {
    const long long kept = totals[3], added = totals[4];
    const long long splits = n - kept;
    totals[0] = kept + added;
    totals[1] = added - 2 * splits;
    totals[2] = splits;
  }
  long long run[2] = {s_warp[0][warp] + incl[0] - sum[0], s_warp[1][warp] + incl[1] - sum[1]};
  for (int64_t b = b0; b < b1; ++b) {
    offsets[2 * b] = run[0];
    offsets[2 * b + 1] = run[1];
    run[0] += counts[2 * b];
    run[1] += counts[2 * b + 1];
  }
}

__device__ __forceinline__ void put(const Sets& S, int64_t n, int64_t stride, int64_t src, int64_t dst,
                                    bool moments) {
#pragma unroll
  for (int pl = 0; pl < 15; ++pl) {
    const int64_t e = (int64_t)pl * n + src, o = (int64_t)pl * stride + dst;
    S.po[o] = __ldg(&S.p[e]);
    S.mo[o] = moments ? __ldg(&S.m[e]) : make_float4(0.f, 0.f, 0.f, 0.f);
    S.vo[o] = moments ? __ldg(&S.v[e]) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// A split child: the parent's planes with the mean moved by R(q / |q|) (s * z) and the
// log-scales lowered by ln 1.6; zero moments.
__device__ __forceinline__ void put_child(const Sets& S, int64_t n, int64_t stride, int64_t src, int64_t dst,
                                          const float* __restrict__ z) {
  const float4 p0 = __ldg(&S.p[src]), p1 = __ldg(&S.p[n + src]), q = __ldg(&S.p[2 * n + src]);
  const float inv = rsqrtf(q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w);
  const float w = q.x * inv, x = q.y * inv, y = q.z * inv, qz = q.w * inv;
  const float sx = expf(p1.x) * z[0], sy = expf(p1.y) * z[1], sz = expf(p1.z) * z[2];
  float4 c0 = p0;
  c0.x += (1.f - 2.f * (y * y + qz * qz)) * sx + 2.f * (x * y - w * qz) * sy + 2.f * (x * qz + w * y) * sz;
  c0.y += 2.f * (x * y + w * qz) * sx + (1.f - 2.f * (x * x + qz * qz)) * sy + 2.f * (y * qz - w * x) * sz;
  c0.z += 2.f * (x * qz - w * y) * sx + 2.f * (y * qz + w * x) * sy + (1.f - 2.f * (x * x + y * y)) * sz;
  const float4 c1 = make_float4(p1.x - kLn16, p1.y - kLn16, p1.z - kLn16, p1.w);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int pl = 0; pl < 15; ++pl) {
    const int64_t o = (int64_t)pl * stride + dst;
    S.po[o] = pl == 0 ? c0 : (pl == 1 ? c1 : __ldg(&S.p[(int64_t)pl * n + src]));
    S.mo[o] = zero;
    S.vo[o] = zero;
  }
}

__global__ void __launch_bounds__(kThreads) k_densify_scatter(const __grid_constant__ Sets S, const float2* stat,
                                                              const float* __restrict__ normals, int64_t n, float thr,
                                                              float lthr, const int64_t* __restrict__ offsets,
                                                              const int64_t* __restrict__ totals, int64_t stride) {
  __shared__ uint32_t s_k[kThreads / 32], s_n[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int kind = i < n ? kind_of(S.p + n, stat, i, thr, lthr) : -1;
  const bool keep = kind == 0 || kind == 1;
  const uint32_t add = kind == 1 ? 1u : (kind == 2 ? 2u : 0u);
  const uint32_t kb = __ballot_sync(0xffffffffu, keep);
  uint32_t ai = add;  // inclusive warp scan of the new counts
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, ai, o);
    if (lane >= o) ai += u;
  }
  if (lane == 31) {
    s_k[warp] = __popc(kb);
    s_n[warp] = ai;
  }
  __syncthreads();
  uint32_t kw = 0, nw = 0;
  for (int w = 0; w < warp; ++w) {
    kw += s_k[w];
    nw += s_n[w];
  }
  if (kind < 0) return;
  if (keep) {
    const int64_t dst = offsets[2 * blockIdx.x] + kw + __popc(kb & ((1u << lane) - 1u));
    if (dst < stride) put(S, n, stride, i, dst, true);
  }
  if (add == 0) return;
  const int64_t dst = totals[3] + offsets[2 * blockIdx.x + 1] + nw + (ai - add);
  if (kind == 1) {
    if (dst < stride) put(S, n, stride, i, dst, false);
    return;
  }
  for (int c = 0; c < 2; ++c)
    if (dst + c < stride) put_child(S, n, stride, i, dst + c, normals + 6 * i + 3 * c);
}

int64_t densify_blocks(int64_t n) { return (n + kThreads - 1) / kThreads; }

}  // namespace

extern "C" size_t gs_densify_workspace_size(int64_t n) {
  if (n < 0) return 0;
  const size_t nb = (size_t)std::max<int64_t>(densify_blocks(n), 1);
  return ((2 * sizeof(uint32_t) * nb + 255) & ~size_t(255)) + 2 * sizeof(int64_t) * nb + 256;
}

extern "C" gs_status gs_densify(const float* params, const float* exp_avg, const float* exp_avg_sq, int64_t n,
                                const float* densify_stat, float grad_threshold, float log_scale_threshold,
                                const float* normals, float* params_out, float* exp_avg_out, float* exp_avg_sq_out,
                                int64_t out_stride, void* workspace, size_t workspace_bytes, int64_t* counts,
                                int64_t* counts_host, void* stream) {
  if (n < 0 || n > (int64_t(1) << 30) || out_stride < 0)
    return gs::set_error(GS_ERR_INVALID, "gs_densify: bad n or out_stride");
  if (!counts || (n > 0 && (!params || !exp_avg || !exp_avg_sq || !densify_stat || !normals || !workspace)) ||
      (out_stride > 0 && (!params_out || !exp_avg_out || !exp_avg_sq_out)))
    return gs::set_error(GS_ERR_INVALID, "gs_densify: NULL pointer");
  if (!gs::aligned8(counts) || (n > 0 && (!gs::aligned16(params) || !gs::aligned16(exp_avg) ||
                                          !gs::aligned16(exp_avg_sq) || !gs::aligned8(densify_stat))) ||
      (out_stride > 0 && (!gs::aligned16(params_out) || !gs::aligned16(exp_avg_out) ||
                          !gs::aligned16(exp_avg_sq_out))) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return gs::set_error(GS_ERR_INVALID, "gs_densify: misaligned pointer");
  cudaStream_t st = gs::as_stream(stream);
  if (n == 0) {
    if (cudaMemsetAsync(counts, 0, 3 * sizeof(int64_t), st) != cudaSuccess) return gs::check_launch("gs_densify");
  } else {
    const size_t need = gs_densify_workspace_size(n);
    if (workspace_bytes < need)
      return gs::set_error(GS_ERR_INVALID, "gs_densify: workspace %zu bytes < %zu needed", workspace_bytes, need);
    const int64_t nb = densify_blocks(n);
    uint32_t* bc = reinterpret_cast<uint32_t*>(workspace);
    char* rest = reinterpret_cast<char*>(workspace) + ((2 * sizeof(uint32_t) * (size_t)nb + 255) & ~size_t(255));
    int64_t* offsets = reinterpret_cast<int64_t*>(rest);
    int64_t* totals = reinterpret_cast<int64_t*>(rest + 2 * sizeof(int64_t) * (size_t)nb);  // [5]
    const float4* p = reinterpret_cast<const float4*>(params);
    const float2* stat = reinterpret_cast<const float2*>(densify_stat);
    k_densify_count<<<(unsigned)nb, kThreads, 0, st>>>(p, stat, n, grad_threshold, log_scale_threshold, bc);
    if (gs_status s = gs::check_launch("gs_densify count")) return s;
    k_densify_scan<<<1, kScan, 0, st>>>(bc, nb, n, offsets, totals);
    if (gs_status s = gs::check_launch("gs_densify scan")) return s;
    if (out_stride > 0) {
      const Sets S{p, reinterpret_cast<const float4*>(exp_avg), reinterpret_cast<const float4*>(exp_avg_sq),
                   reinterpret_cast<float4*>(params_out), reinterpret_cast<float4*>(exp_avg_out),
                   reinterpret_cast<float4*>(exp_avg_sq_out)};
      k_densify_scatter<<<(unsigned)nb, kThreads, 0, st>>>(S, stat, normals, n, grad_threshold, log_scale_threshold,
                                                           offsets, totals, out_stride);
      if (gs_status s = gs::check_launch("gs_densify scatter")) return s;
    }
    if (cudaMemcpyAsync(counts, totals, 3 * sizeof(int64_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return gs::check_launch("gs_densify counts");
  }
  if (!counts_host) return GS_OK;
  if (cudaMemcpyAsync(counts_host, counts, 3 * sizeof(int64_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return gs::check_launch("gs_densify readback");
  if (out_stride > 0 && counts_host[0] > out_stride)
    return gs::set_error(GS_ERR_CAPACITY, "gs_densify: %lld Gaussians exceed the output stride %lld",
                         (long long)counts_host[0], (long long)out_stride);
  return GS_OK;
}
