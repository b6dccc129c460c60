// Visible sets with pairwise overlaps (gs_visible_sets) and the visible-only batched Adam
// update (gs_sparse_adam).
//
// Odin summary, "研究背景与动机": every view renders, backpropagates and updates only the
// primitives it sees; §1: Jaccard weight |Pi n Pj| / |Pi u Pj| (0 for an empty union).
// Grendel-GS notes §4.2: lr' = lr sqrt(batch), beta' = beta^batch.
//
// Visible sets are built from one bit per Gaussian per view (a warp ballot over the radius
// of 32 consecutive Gaussians), so every later pass reads N/8 bytes per view: counts and
// the ascending index lists come from a block-count / scan / write compaction, the union is
// the OR of the views' words, and all B(B+1)/2 intersections are popcounts of ANDed words
// staged per CTA in shared memory.
#include <cmath>

#include "common.cuh"

namespace {

constexpr int kMaxViews = 64;
constexpr int kWordsPerBlock = 256;  // one thread per 32-bit word

struct ViewPtrs {
  const float* q[kMaxViews];
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct VisWs {
  uint32_t* bits;     // [B + 1][nwords]; set B is the union
  uint32_t* blkcnt;   // [B + 1][nblk] -> exclusive prefix after the scan
  uint32_t* totals;   // [B + 1]
};

size_t vis_carve(VisWs* w, char* base, int B, int64_t n) {
  const int64_t nwords = (n + 31) / 32;
  const int64_t nblk = (nwords + kWordsPerBlock - 1) / kWordsPerBlock;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* p = base ? base + off : nullptr;
    off += align256(bytes);
    return p;
  };
  char* b = take(sizeof(uint32_t) * (size_t)(B + 1) * (size_t)std::max<int64_t>(nwords, 1));
  char* c = take(sizeof(uint32_t) * (size_t)(B + 1) * (size_t)std::max<int64_t>(nblk, 1));
  char* t = take(sizeof(uint32_t) * (size_t)(B + 1));
  if (w) {
    w->bits = reinterpret_cast<uint32_t*>(b);
    w->blkcnt = reinterpret_cast<uint32_t*>(c);
    w->totals = reinterpret_cast<uint32_t*>(t);
  }
  return off;
}

// bits[b][word]: ballot of radius > 0 over 32 consecutive Gaussians
__global__ void __launch_bounds__(256) k_vis_bits(ViewPtrs views, int64_t n, int64_t nwords, uint32_t* bits) {
  const int b = blockIdx.y;
  const int64_t word = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (word >= nwords) return;
  const int64_t i = word * 32 + lane;
  bool vis = false;
  if (i < n) vis = __float_as_int(__ldg(reinterpret_cast<const float4*>(views.q[b]) + n + i).w) > 0;
  const uint32_t m = __ballot_sync(0xffffffffu, vis);
  if (lane == 0) bits[(int64_t)b * nwords + word] = m;
}

// union words + per-block popcounts of every set
__global__ void __launch_bounds__(kWordsPerBlock) k_vis_count(int B, int64_t nwords, int64_t nblk, uint32_t* bits,
                                                              uint32_t* blkcnt) {
  __shared__ uint32_t s[kWordsPerBlock / 32];
  const int set = blockIdx.y;
  const int64_t word = (int64_t)blockIdx.x * kWordsPerBlock + threadIdx.x;
  uint32_t m = 0;
  if (word < nwords) {
    if (set < B) {
      m = bits[(int64_t)set * nwords + word];
    } else {
      for (int b = 0; b < B; ++b) m |= bits[(int64_t)b * nwords + word];
      bits[(int64_t)B * nwords + word] = m;
    }
  }
  uint32_t c = __popc(m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kWordsPerBlock / 32; ++w) t += s[w];
    blkcnt[(int64_t)set * nblk + blockIdx.x] = t;
  }
}

// exclusive scan of the block counts of one set (one CTA per set), totals, offsets
__global__ void __launch_bounds__(1024) k_vis_scan(int B, int64_t nblk, uint32_t* blkcnt, uint32_t* totals) {
  __shared__ uint32_t s_warp[32];
  __shared__ uint32_t s_carry;
  const int set = blockIdx.x;
  uint32_t* c = blkcnt + (int64_t)set * nblk;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_carry = 0;
  __syncthreads();
  for (int64_t b0 = 0; b0 < nblk; b0 += 1024) {
    const int64_t i = b0 + threadIdx.x;
    const uint32_t v = i < nblk ? c[i] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    uint32_t woff = 0, tot = 0;
    for (int w = 0; w < 32; ++w) {
      if (w < warp) woff += s_warp[w];
      tot += s_warp[w];
    }
    const uint32_t carry = s_carry;
    if (i < nblk) c[i] = carry + woff + incl - v;
    __syncthreads();
    if (threadIdx.x == 0) s_carry = carry + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) totals[set] = s_carry;
}

__global__ void k_vis_offsets(int B, const uint32_t* totals, int64_t* offsets, int64_t* n_union) {
  if (threadIdx.x == 0 && blockIdx.x == 0) {
    int64_t run = 0;
    for (int b = 0; b < B; ++b) {
      offsets[b] = run;
      run += totals[b];
    }
    offsets[B] = run;
    *n_union = totals[B];
  }
}

// ascending index lists: each word's bits at its block prefix + warp prefix
__global__ void __launch_bounds__(kWordsPerBlock) k_vis_write(int B, int64_t nwords, int64_t nblk,
                                                              const uint32_t* bits, const uint32_t* blkcnt,
                                                              const int64_t* offsets, uint32_t* indices,
                                                              uint32_t* union_idx) {
  // each warp's indices (up to 32 per lane, in order) are staged in shared memory and then
  // written to the output as consecutive words, instead of every lane storing its own run
  __shared__ uint32_t s[kWordsPerBlock / 32];
  __shared__ uint32_t stage[kWordsPerBlock / 32][32 * 32];
  const int set = blockIdx.y;
  const int64_t word = (int64_t)blockIdx.x * kWordsPerBlock + threadIdx.x;
  const uint32_t m = word < nwords ? bits[(int64_t)set * nwords + word] : 0u;
  const uint32_t c = __popc(m);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s[warp] = incl;
  __syncthreads();
  uint32_t woff = 0;
  for (int w = 0; w < warp; ++w) woff += s[w];
  const uint32_t wtotal = __shfl_sync(0xffffffffu, incl, 31);
  uint32_t* st = stage[warp];
  uint32_t k = incl - c;
  uint32_t mm = m;
  while (mm) {
    const int bit = __ffs(mm) - 1;
    mm &= mm - 1;
    st[k++] = (uint32_t)(word * 32 + bit);
  }
  __syncwarp();
  uint32_t* out = (set < B ? indices + offsets[set] : union_idx) + blkcnt[(int64_t)set * nblk + blockIdx.x] + woff;
  for (uint32_t j = lane; j < wtotal; j += 32) out[j] = st[j];
}

__global__ void __launch_bounds__(256) k_vis_inter(int B, int64_t nwords, const uint32_t* bits,
                                                   unsigned long long* inter) {
  extern __shared__ uint32_t s_words[];  // [B][256]
  const int64_t w0 = (int64_t)blockIdx.x * 256;
  for (int b = 0; b < B; ++b) {
    const int64_t w = w0 + threadIdx.x;
    s_words[b * 256 + threadIdx.x] = w < nwords ? bits[(int64_t)b * nwords + w] : 0u;
  }
  __syncthreads();
  const int npairs = B * (B + 1) / 2;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    int i = 0, rem = p;
    while (rem >= B - i) {
      rem -= B - i;
      ++i;
    }
    const int j = i + rem;
    uint32_t acc = 0;
    const uint32_t* a = s_words + i * 256;
    const uint32_t* c = s_words + j * 256;
    for (int k = 0; k < 256; ++k) acc += __popc(a[k] & c[k]);
    if (acc) atomicAdd(&inter[i * B + j], (unsigned long long)acc);
  }
}

__global__ void k_vis_jaccard(int B, int64_t* inter, float* jac) {
  const int i = blockIdx.x, j = threadIdx.x;
  if (i >= B || j >= B) return;
  // upper triangle holds the sums; mirror it
  const int64_t v = i <= j ? inter[i * B + j] : inter[j * B + i];
  const int64_t ni = inter[i * B + i], nj = inter[j * B + j];
  __syncthreads();
  inter[i * B + j] = v;
  const int64_t un = ni + nj - v;
  jac[i * B + j] = un == 0 ? 0.f : (float)((double)v / (double)un);
}

// ------------------------------------------------------------------ Adam
__global__ void __launch_bounds__(256) k_sparse_adam(float4* __restrict__ p, float4* __restrict__ g,
                                                     float4* __restrict__ m, float4* __restrict__ v, int64_t n,
                                                     const uint32_t* __restrict__ idx, const int64_t* n_idx,
                                                     int64_t max_idx, float b1, float b2, float lr_c, float ibc2,
                                                     float eps, const int64_t* counts, int n_counts) {
  for (int c = 0; c < n_counts; ++c)
    if (counts[2 * c + 1] != 0) return;  // a view of this batch overflowed its binning
  const int64_t nu = min(*n_idx, max_idx);
  const int plane = blockIdx.y;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < nu; u += stride) {
    const int64_t e = (int64_t)plane * n + __ldg(&idx[u]);
    const float4 gg = g[e];
    float4 mm = m[e], vv = v[e], pp = p[e];
    const float ga[4] = {gg.x, gg.y, gg.z, gg.w};
    float* ma = &mm.x;
    float* va = &vv.x;
    float* pa = &pp.x;
#pragma unroll
    for (int l = 0; l < 4; ++l) {
      ma[l] = b1 * ma[l] + (1.f - b1) * ga[l];
      va[l] = b2 * va[l] + (1.f - b2) * ga[l] * ga[l];
      // lr_c = lr' / (1 - beta1'^step), ibc2 = 1 / (1 - beta2'^step): host-computed factors and
      // one fast division instead of two IEEE divisions (a few ulp of the update)
      pa[l] -= __fdividef(lr_c * ma[l], sqrtf(va[l] * ibc2) + eps);
    }
    p[e] = pp;
    m[e] = mm;
    v[e] = vv;
    g[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

}  // namespace

extern "C" size_t gs_visible_sets_workspace_size(int batch, int64_t n) {
  if (batch < 1 || batch > kMaxViews || n < 0) return 0;
  return vis_carve(nullptr, nullptr, batch, n);
}

extern "C" gs_status gs_visible_sets(const float* const* proj_per_view, int batch, int64_t n, void* workspace,
                                     size_t workspace_bytes, int64_t* offsets, uint32_t* indices,
                                     uint32_t* union_idx, int64_t* n_union, int64_t* inter, float* jaccard,
                                     const uint32_t* visible_bits, int64_t bits_stride, void* stream) {
  if (batch < 1 || batch > kMaxViews) return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: batch must be 1..64");
  if (n < 0 || n >= (int64_t(1) << 32)) return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: bad n");
  if ((!proj_per_view && !visible_bits) || !workspace || !offsets || !n_union || !inter || !jaccard ||
      (n > 0 && (!indices || !union_idx)))
    return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: NULL pointer");
  if (visible_bits && bits_stride < (n + 31) / 32)
    return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: bits_stride %lld < ceil(n / 32)", (long long)bits_stride);
  const size_t need = vis_carve(nullptr, nullptr, batch, n);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: workspace must be 256-byte aligned");
  ViewPtrs vp{};
  for (int b = 0; b < batch && !visible_bits; ++b) {
    if (n > 0 && (!proj_per_view[b] || !gs::aligned16(proj_per_view[b])))
      return gs::set_error(GS_ERR_INVALID, "gs_visible_sets: view %d proj NULL or misaligned", b);
    vp.q[b] = proj_per_view[b];
  }
  VisWs w;
  vis_carve(&w, reinterpret_cast<char*>(workspace), batch, n);
  cudaStream_t st = gs::as_stream(stream);
  const int64_t nwords = (n + 31) / 32;
  const int64_t nblk = (nwords + kWordsPerBlock - 1) / kWordsPerBlock;
  if (cudaMemsetAsync(inter, 0, sizeof(int64_t) * batch * batch, st) != cudaSuccess)
    return gs::check_launch("gs_visible_sets memset");
  if (n > 0) {
    if (visible_bits) {  // the caller's bitsets: copied into the workspace's sets
      if (cudaMemcpy2DAsync(w.bits, sizeof(uint32_t) * nwords, visible_bits, sizeof(uint32_t) * bits_stride,
                            sizeof(uint32_t) * nwords, (size_t)batch, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return gs::check_launch("gs_visible_sets bitsets");
    } else {
      dim3 gb((unsigned)((nwords * 32 + 255) / 256), (unsigned)batch);
      k_vis_bits<<<gb, 256, 0, st>>>(vp, n, nwords, w.bits);
    }
    dim3 gc((unsigned)nblk, (unsigned)(batch + 1));
    k_vis_count<<<gc, kWordsPerBlock, 0, st>>>(batch, nwords, nblk, w.bits, w.blkcnt);
  } else {
    cudaMemsetAsync(w.totals, 0, sizeof(uint32_t) * (batch + 1), st);
  }
  if (n > 0) k_vis_scan<<<batch + 1, 1024, 0, st>>>(batch, nblk, w.blkcnt, w.totals);
  k_vis_offsets<<<1, 32, 0, st>>>(batch, w.totals, offsets, n_union);
  if (gs_status s = gs::check_launch("gs_visible_sets scan")) return s;
  if (n > 0) {
    dim3 gw((unsigned)nblk, (unsigned)(batch + 1));
    k_vis_write<<<gw, kWordsPerBlock, 0, st>>>(batch, nwords, nblk, w.bits, w.blkcnt, offsets, indices, union_idx);
    const size_t smem = sizeof(uint32_t) * 256 * batch;
    const cudaError_t attr = gs::max_dynamic_smem((const void*)k_vis_inter, 256 * 4 * kMaxViews);
    if (attr != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_visible_sets: %s", cudaGetErrorString(attr));
    k_vis_inter<<<(unsigned)((nwords + 255) / 256), 256, smem, st>>>(batch, nwords, w.bits,
                                                                     reinterpret_cast<unsigned long long*>(inter));
  }
  k_vis_jaccard<<<batch, batch, 0, st>>>(batch, inter, jaccard);
  return gs::check_launch("gs_visible_sets");
}

extern "C" gs_status gs_sparse_adam(float* params, float* grads, float* exp_avg, float* exp_avg_sq, int64_t n,
                                    const uint32_t* idx, const int64_t* n_idx, int64_t max_idx, float lr,
                                    float beta1, float beta2, float eps, int batch, int64_t step,
                                    const int64_t* counts, int n_counts, void* stream) {
  if (n < 0 || max_idx < 0 || max_idx > n) return gs::set_error(GS_ERR_INVALID, "gs_sparse_adam: bad n / max_idx");
  if (batch < 1 || step < 1) return gs::set_error(GS_ERR_INVALID, "gs_sparse_adam: batch and step must be >= 1");
  if (n == 0 || max_idx == 0) return GS_OK;
  if (!params || !grads || !exp_avg || !exp_avg_sq || !idx || !n_idx || (n_counts > 0 && !counts))
    return gs::set_error(GS_ERR_INVALID, "gs_sparse_adam: NULL pointer");
  if (n_counts < 0 || !counts) n_counts = 0;
  if (!gs::aligned16(params) || !gs::aligned16(grads) || !gs::aligned16(exp_avg) || !gs::aligned16(exp_avg_sq))
    return gs::set_error(GS_ERR_INVALID, "gs_sparse_adam: planes must be 16-byte aligned");
  // batch scaling rule: lr sqrt(b), beta^b; bias corrections with the scaled betas
  const double b1 = std::pow((double)beta1, batch), b2 = std::pow((double)beta2, batch);
  const double lr_b = (double)lr * std::sqrt((double)batch);
  const double bc1 = 1.0 - std::pow(b1, (double)step), bc2 = 1.0 - std::pow(b2, (double)step);
  const int64_t per_plane = std::min<int64_t>(max_idx, (int64_t)gs::num_sms() * 8 * 256);
  dim3 grid((unsigned)((per_plane + 255) / 256), 15);
  k_sparse_adam<<<grid, 256, 0, gs::as_stream(stream)>>>(
      reinterpret_cast<float4*>(params), reinterpret_cast<float4*>(grads), reinterpret_cast<float4*>(exp_avg),
      reinterpret_cast<float4*>(exp_avg_sq), n, idx, n_idx, max_idx, (float)b1, (float)b2, (float)(lr_b / bc1),
      (float)(1.0 / bc2), eps, counts, n_counts);
  return gs::check_launch("gs_sparse_adam");
}
