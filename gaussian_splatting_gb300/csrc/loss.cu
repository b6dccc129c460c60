// L1 + SSIM image loss and its gradient in one fused pass (gs_loss).
//
// "Loss" step of the Grendel-GS training flow (训练流程: L1 + SSIM).  Each CTA owns a 32x32
// output tile of one channel.  It loads the image and target with a 10-pixel halo, blurs
// the five SSIM statistics (x, y, x^2, y^2, xy) separably with the 11-tap window over the
// tile plus a 5-pixel halo, forms the SSIM map and its three partial derivatives there
// (zero outside the image), and blurs those back onto the tile (the window is symmetric,
// so the adjoint of the zero-padded window sum is the same window sum).  Nothing but the
// per-CTA partial sums of SSIM and |x - y| goes to global scratch; a last one-CTA kernel
// reduces them in a fixed order.
#include <cmath>

#include "common.cuh"

namespace {

constexpr int kOut = 32;               // output tile edge
constexpr int kR = 5;                  // window radius
constexpr int kMid = kOut + 2 * kR;    // 42: SSIM map region
constexpr int kIn = kOut + 4 * kR;     // 52: input region
constexpr int kThreads = 256;

struct Window {
  float w[11];
};

struct LossSmem {
  // phase A: inputs; phase B: derivative maps (aliases the inputs)
  union {
    struct {
      float x[kIn][kIn];
      float y[kIn][kIn];
    } in;
    float d[3][kMid][kMid];
  } u1;
  // phase A: horizontal blur of 5 statistics; phase C: horizontal blur of 3 maps
  union {
    float h5[5][kIn][kMid];
    float h3[3][kMid][kOut + 1];  // padded row: the row-blocked writes of phase C hit distinct banks
  } u2;
  float core[2][kOut][kOut];  // image and target on the output tile
  float red[2][kThreads / 32];
};

// Register-blocked window sums: a thread produces R consecutive outputs along the blur
// direction from R + 10 loaded inputs (sliding window), instead of 11 loads per output.
constexpr int kRA = 6;  // horizontal blur of the statistics: 42 = 7 x 6 outputs per row
constexpr int kRB = 7;  // vertical blur of the statistics: 42 = 6 x 7 outputs per column
constexpr int kRC = 4;  // horizontal blur of the derivative maps: 32 = 8 x 4 per row
constexpr int kRD = 4;  // vertical blur of the derivative maps: 32 = 8 x 4 per column

__global__ void __launch_bounds__(kThreads) k_loss_fused(const float* __restrict__ img, const float* __restrict__ tgt,
                                                          int W, int H, Window win, float w_l1, float w_ssim,
                                                          float scale, float inv_n, float* __restrict__ dimg,
                                                          float* __restrict__ partials) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  LossSmem& S = *reinterpret_cast<LossSmem*>(smem_raw);
  const int ch = blockIdx.z;
  const int ox = blockIdx.x * kOut, oy = blockIdx.y * kOut;
  const int64_t P = (int64_t)W * H;
  const float* X = img + ch * P;
  const float* Y = tgt + ch * P;
  const int tid = threadIdx.x;
  float w[11];
#pragma unroll
  for (int t = 0; t < 11; ++t) w[t] = win.w[t];
  // ---- A: load with 10-px halo (zero outside the image); all loads of a thread in flight
  // together, the output tile's own pixels also kept aside for the last stage
  constexpr int kLoadIters = (kIn * kIn + kThreads - 1) / kThreads;
  {
    float xv[kLoadIters], yv[kLoadIters];
#pragma unroll
    for (int it = 0; it < kLoadIters; ++it) {
      const int e = tid + it * kThreads;
      const int r = e / kIn, c = e % kIn;
      const int gy = oy - 2 * kR + r, gx = ox - 2 * kR + c;
      xv[it] = yv[it] = 0.f;
      if (e < kIn * kIn && gx >= 0 && gx < W && gy >= 0 && gy < H) {
        xv[it] = __ldg(&X[(int64_t)gy * W + gx]);
        yv[it] = __ldg(&Y[(int64_t)gy * W + gx]);
      }
    }
#pragma unroll
    for (int it = 0; it < kLoadIters; ++it) {
      const int e = tid + it * kThreads;
      if (e < kIn * kIn) {
        const int r = e / kIn, c = e % kIn;
        S.u1.in.x[r][c] = xv[it];
        S.u1.in.y[r][c] = yv[it];
        const int cr = r - 2 * kR, cc = c - 2 * kR;
        if (cr >= 0 && cr < kOut && cc >= 0 && cc < kOut) {
          S.core[0][cr][cc] = xv[it];
          S.core[1][cr][cc] = yv[it];
        }
      }
    }
  }
  __syncthreads();
  // horizontal window sums of x, y, x^2, y^2, xy: 52 rows x 42 columns, kRA per thread
  constexpr int kSegA = kMid / kRA;
  for (int item = tid; item < kIn * kSegA; item += kThreads) {
    const int r = item / kSegA, c0 = (item % kSegA) * kRA;
    float a[5][kRA];
#pragma unroll
    for (int q = 0; q < kRA; ++q) a[0][q] = a[1][q] = a[2][q] = a[3][q] = a[4][q] = 0.f;
#pragma unroll
    for (int e = 0; e < kRA + 10; ++e) {
      const float xv = S.u1.in.x[r][c0 + e], yv = S.u1.in.y[r][c0 + e];
      const float xx = xv * xv, yy = yv * yv, xy = xv * yv;
#pragma unroll
      for (int q = 0; q < kRA; ++q) {
        const int t = e - q;  // tap index of input e for output q
        if (t >= 0 && t < 11) {
          a[0][q] = fmaf(w[t], xv, a[0][q]);
          a[1][q] = fmaf(w[t], yv, a[1][q]);
          a[2][q] = fmaf(w[t], xx, a[2][q]);
          a[3][q] = fmaf(w[t], yy, a[3][q]);
          a[4][q] = fmaf(w[t], xy, a[4][q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRA; ++q)
#pragma unroll
      for (int m = 0; m < 5; ++m) S.u2.h5[m][r][c0 + q] = a[m][q];
  }
  __syncthreads();
  // ---- B: vertical window sums -> SSIM statistics on the 42x42 region; map + derivatives
  constexpr float C1 = 0.01f * 0.01f, C2 = 0.03f * 0.03f;
  constexpr int kSegB = kMid / kRB;
  constexpr int kItemsB = kMid * kSegB;                         // 252
  constexpr int kRoundsB = (kItemsB + kThreads - 1) / kThreads;  // 1
  float ssim_sum = 0.f;
  float dv[kRoundsB][kRB][3];
#pragma unroll
  for (int rd = 0; rd < kRoundsB; ++rd) {
    const int item = tid + rd * kThreads;
#pragma unroll
    for (int q = 0; q < kRB; ++q) dv[rd][q][0] = dv[rd][q][1] = dv[rd][q][2] = 0.f;
    if (item >= kItemsB) continue;
    const int c = item % kMid, r0 = (item / kMid) * kRB;
    float a[5][kRB];
#pragma unroll
    for (int q = 0; q < kRB; ++q) a[0][q] = a[1][q] = a[2][q] = a[3][q] = a[4][q] = 0.f;
#pragma unroll
    for (int e = 0; e < kRB + 10; ++e) {
      float v[5];
#pragma unroll
      for (int m = 0; m < 5; ++m) v[m] = S.u2.h5[m][r0 + e][c];
#pragma unroll
      for (int q = 0; q < kRB; ++q) {
        const int t = e - q;
        if (t >= 0 && t < 11) {
#pragma unroll
          for (int m = 0; m < 5; ++m) a[m][q] = fmaf(w[t], v[m], a[m][q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRB; ++q) {
      const int r = r0 + q;
      const int gy = oy - kR + r, gx = ox - kR + c;
      if (gx >= 0 && gx < W && gy >= 0 && gy < H) {
        const float mx = a[0][q], my = a[1][q];
        const float sxx = a[2][q] - mx * mx, syy = a[3][q] - my * my, sxy = a[4][q] - mx * my;
        const float A1 = 2.f * mx * my + C1, A2 = 2.f * sxy + C2;
        const float B1 = mx * mx + my * my + C1, B2 = sxx + syy + C2;
        // two fast reciprocals (B1 >= C1, B2 >= C2 - rounding: far from zero) serve all four quotients
        const float iB1 = __fdividef(1.f, B1), iB2 = __fdividef(1.f, B2);
        const float iB = iB1 * iB2;
        const float Sv = A1 * A2 * iB;
        dv[rd][q][0] = 2.f * my * (A2 - A1) * iB - 2.f * mx * Sv * (iB1 - iB2);  // dS/dmu_x
        dv[rd][q][1] = -Sv * iB2;                                                  // dS/dE[x^2]
        dv[rd][q][2] = 2.f * A1 * iB;                                              // dS/dE[xy]
        if (r >= kR && r < kR + kOut && c >= kR && c < kR + kOut) ssim_sum += Sv;
      }
    }
  }
  __syncthreads();  // inputs no longer needed: the derivative maps overwrite them
#pragma unroll
  for (int rd = 0; rd < kRoundsB; ++rd) {
    const int item = tid + rd * kThreads;
    if (item >= kItemsB) continue;
    const int c = item % kMid, r0 = (item / kMid) * kRB;
#pragma unroll
    for (int q = 0; q < kRB; ++q)
#pragma unroll
      for (int m = 0; m < 3; ++m) S.u1.d[m][r0 + q][c] = dv[rd][q][m];
  }
  __syncthreads();
  // ---- C: horizontal window sums of the three derivative maps onto the output columns
  constexpr int kSegC = kOut / kRC;
  for (int item = tid; item < kMid * kSegC; item += kThreads) {
    const int r = item / kSegC, c0 = (item % kSegC) * kRC;
    float a[3][kRC];
#pragma unroll
    for (int q = 0; q < kRC; ++q) a[0][q] = a[1][q] = a[2][q] = 0.f;
#pragma unroll
    for (int e = 0; e < kRC + 10; ++e) {
      float v[3];
#pragma unroll
      for (int m = 0; m < 3; ++m) v[m] = S.u1.d[m][r][c0 + e];
#pragma unroll
      for (int q = 0; q < kRC; ++q) {
        const int t = e - q;
        if (t >= 0 && t < 11) {
#pragma unroll
          for (int m = 0; m < 3; ++m) a[m][q] = fmaf(w[t], v[m], a[m][q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kRC; ++q)
#pragma unroll
      for (int m = 0; m < 3; ++m) S.u2.h3[m][r][c0 + q] = a[m][q];
  }
  __syncthreads();
  // ---- D: vertical window sums, combine with the L1 term, write dL/dx
  float l1_sum = 0.f;
  constexpr int kSegD = kOut / kRD;
  for (int item = tid; item < kOut * kSegD; item += kThreads) {
    const int c = item % kOut, r0 = (item / kOut) * kRD;
    float a[3][kRD];
#pragma unroll
    for (int q = 0; q < kRD; ++q) a[0][q] = a[1][q] = a[2][q] = 0.f;
#pragma unroll
    for (int e = 0; e < kRD + 10; ++e) {
      float v[3];
#pragma unroll
      for (int m = 0; m < 3; ++m) v[m] = S.u2.h3[m][r0 + e][c];
#pragma unroll
      for (int q = 0; q < kRD; ++q) {
        const int t = e - q;
        if (t >= 0 && t < 11) {
#pragma unroll
          for (int m = 0; m < 3; ++m) a[m][q] = fmaf(w[t], v[m], a[m][q]);
        }
      }
    }
    const int gx = ox + c;
#pragma unroll
    for (int q = 0; q < kRD; ++q) {
      const int gy = oy + r0 + q;
      if (gx >= W || gy >= H) continue;
      const int64_t g = (int64_t)gy * W + gx;
      const float xv = S.core[0][r0 + q][c], yv = S.core[1][r0 + q][c];
      const float diff = xv - yv;
      l1_sum += fabsf(diff);
      const float sgn = diff > 0.f ? 1.f : (diff < 0.f ? -1.f : 0.f);
      const float dssim = a[0][q] + 2.f * xv * a[1][q] + yv * a[2][q];
      dimg[ch * P + g] = scale * inv_n * (w_l1 * sgn - w_ssim * dssim);
    }
  }
  // ---- fixed-order block reduction of the two sums
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ssim_sum += __shfl_xor_sync(0xffffffffu, ssim_sum, o);
    l1_sum += __shfl_xor_sync(0xffffffffu, l1_sum, o);
  }
  if (lane == 0) {
    S.red[0][warp] = ssim_sum;
    S.red[1][warp] = l1_sum;
  }
  __syncthreads();
  if (tid == 0) {
    float a = 0.f, b = 0.f;
    for (int w2 = 0; w2 < kThreads / 32; ++w2) {
      a += S.red[0][w2];
      b += S.red[1][w2];
    }
    const int64_t blk = ((int64_t)blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
    partials[2 * blk] = a;
    partials[2 * blk + 1] = b;
  }
}

__global__ void __launch_bounds__(256) k_loss_final(const float* __restrict__ partials, int64_t nblk, float w_l1,
                                                     float w_ssim, float scale, double inv_n, float* loss,
                                                     int accumulate) {
  __shared__ double s[2][256];
  double a = 0.0, b = 0.0;
  for (int64_t i = threadIdx.x; i < nblk; i += 256) {
    a += (double)partials[2 * i];
    b += (double)partials[2 * i + 1];
  }
  s[0][threadIdx.x] = a;
  s[1][threadIdx.x] = b;
  __syncthreads();
  for (int o = 128; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) {
      s[0][threadIdx.x] += s[0][threadIdx.x + o];
      s[1][threadIdx.x] += s[1][threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double ssim = s[0][0] * inv_n, l1 = s[1][0] * inv_n;
    const float v = (float)((double)scale * ((double)w_l1 * l1 + (double)w_ssim * (1.0 - ssim)));
    *loss = accumulate ? *loss + v : v;
  }
}

int64_t loss_blocks(int W, int H) {
  return (int64_t)((W + kOut - 1) / kOut) * ((H + kOut - 1) / kOut) * 3;
}

Window make_window() {
  double h[11], s = 0;
  for (int k = 0; k < 11; ++k) {
    h[k] = std::exp(-double((k - 5) * (k - 5)) / (2.0 * 1.5 * 1.5));
    s += h[k];
  }
  Window w;
  for (int k = 0; k < 11; ++k) w.w[k] = (float)(h[k] / s);
  return w;
}

}  // namespace

extern "C" size_t gs_loss_workspace_size(int width, int height) {
  if (width <= 0 || height <= 0) return 0;
  return sizeof(float) * 2 * (size_t)loss_blocks(width, height);
}

extern "C" gs_status gs_loss(const float* image, const float* target, int width, int height, float w_l1,
                             float w_ssim, float scale, float* loss_dev, int accumulate, float* dL_dimage,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (width <= 0 || height <= 0 || width > 32768 || height > 32768)
    return gs::set_error(GS_ERR_INVALID, "gs_loss: bad image size %d x %d", width, height);
  if (!image || !target || !loss_dev || !dL_dimage || !workspace)
    return gs::set_error(GS_ERR_INVALID, "gs_loss: NULL pointer");
  if (!gs::aligned8(workspace)) return gs::set_error(GS_ERR_INVALID, "gs_loss: misaligned workspace");
  const size_t need = gs_loss_workspace_size(width, height);
  if (workspace_bytes < need)
    return gs::set_error(GS_ERR_INVALID, "gs_loss: workspace %zu bytes < %zu needed", workspace_bytes, need);
  const cudaError_t attr = gs::max_dynamic_smem((const void*)k_loss_fused, (int)sizeof(LossSmem));
  if (attr != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_loss: %s", cudaGetErrorString(attr));
  cudaStream_t st = gs::as_stream(stream);
  const double n = 3.0 * (double)width * (double)height;
  dim3 grid((width + kOut - 1) / kOut, (height + kOut - 1) / kOut, 3);
  float* partials = reinterpret_cast<float*>(workspace);
  k_loss_fused<<<grid, kThreads, sizeof(LossSmem), st>>>(image, target, width, height, make_window(), w_l1, w_ssim,
                                                         scale, (float)(1.0 / n), dL_dimage, partials);
  if (gs_status s = gs::check_launch("gs_loss")) return s;
  k_loss_final<<<1, 256, 0, st>>>(partials, loss_blocks(width, height), w_l1, w_ssim, scale, 1.0 / n, loss_dev,
                                  accumulate);
  return gs::check_launch("gs_loss final");
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of gs_loss.
//
// gs_loss needs a small caller workspace for its per-block partial sums.  Some callers cannot
// hand one out: code whose device memory is owned by another allocator under a fixed budget,
// or code that must not call cudaMalloc / cudaFree because those calls can synchronise the
// whole device.  gs_loss_noalloc keeps the partial sums in a fixed array that lives in this
// library's own device image instead, so it needs no workspace and allocates nothing.
//
// The array holds at most kNoAllocMaxBlocks partial-sum pairs (512 KB; every GPU that loads
// the library keeps it until the process exits): images with
// ceil(W/32) * ceil(H/32) * 3 <= 65536, e.g. up to 4096 x 4096.  Larger images are rejected.
// All calls share the one array: two calls that overlap on the GPU (different streams, no
// ordering between them) race on it.  Every block of a call rewrites its own pair before the
// final reduction reads it, so nothing has to be cleared between calls.
namespace {

constexpr int64_t kNoAllocMaxBlocks = 65536;

static __device__ __align__(256) float g_loss_scratch[2 * kNoAllocMaxBlocks];

// Device address of g_loss_scratch on the current device.  Host code cannot use the symbol
// itself (in host code it names a host-side stand-in), so the address is asked for with the
// device current.  It is asked for on every call -- a host-side lookup that allocates nothing
// -- rather than cached: a cached address would outlive a cudaDeviceReset, after which the
// library's device image is loaded again at another address.  The first call on a device
// also loads the library's device code there, so that first call should come before any
// stream capture.
gs_status scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_loss_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_loss_scratch);
  if (e != cudaSuccess || !p)
    return gs::set_error(GS_ERR_CUDA, "gs_loss_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
  *out = reinterpret_cast<float*>(p);
  return GS_OK;
}

}  // namespace

extern "C" gs_status gs_loss_noalloc(const float* image, const float* target, int width, int height, float w_l1,
                                     float w_ssim, float scale, float* loss_dev, int accumulate, float* dL_dimage,
                                     void* stream) {
  if (width <= 0 || height <= 0 || width > 32768 || height > 32768)
    return gs::set_error(GS_ERR_INVALID, "gs_loss_noalloc: bad image size %d x %d", width, height);
  if (!image || !target || !loss_dev || !dL_dimage) return gs::set_error(GS_ERR_INVALID, "gs_loss_noalloc: NULL pointer");
  const int64_t nblk = loss_blocks(width, height);
  if (nblk > kNoAllocMaxBlocks)
    return gs::set_error(GS_ERR_INVALID,
                         "gs_loss_noalloc: %d x %d needs %lld partial sums, the built-in scratch holds %lld "
                         "(ceil(W/32) * ceil(H/32) * 3 must be <= %lld); use gs_loss with a workspace",
                         width, height, (long long)nblk, (long long)kNoAllocMaxBlocks, (long long)kNoAllocMaxBlocks);
  float* partials = nullptr;
  if (gs_status s = scratch_address(&partials)) return s;
  const cudaError_t attr = gs::max_dynamic_smem((const void*)k_loss_fused, (int)sizeof(LossSmem));
  if (attr != cudaSuccess) return gs::set_error(GS_ERR_CUDA, "gs_loss_noalloc: %s", cudaGetErrorString(attr));
  cudaStream_t st = gs::as_stream(stream);
  const double n = 3.0 * (double)width * (double)height;
  dim3 grid((width + kOut - 1) / kOut, (height + kOut - 1) / kOut, 3);
  k_loss_fused<<<grid, kThreads, sizeof(LossSmem), st>>>(image, target, width, height, make_window(), w_l1, w_ssim,
                                                         scale, (float)(1.0 / n), dL_dimage, partials);
  if (gs_status s = gs::check_launch("gs_loss_noalloc")) return s;
  k_loss_final<<<1, 256, 0, st>>>(partials, nblk, w_l1, w_ssim, scale, 1.0 / n, loss_dev, accumulate);
  return gs::check_launch("gs_loss_noalloc final");
}
