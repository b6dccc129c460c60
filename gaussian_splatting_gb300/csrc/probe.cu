// FP32 throughput probe (gs_probe_ffma): the measured denominator for the compositing and
// loss kernels, whose bound is plain FP32 arithmetic.  Eight independent FFMA chains per
// thread at full occupancy; the caller times the launch.
#include "common.cuh"

namespace {

__global__ void __launch_bounds__(256) k_probe_ffma(float* __restrict__ out, int iters, float a, float b) {
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = (float)(threadIdx.x + j);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = fmaf(v[j], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += v[j];
  out[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace

extern "C" gs_status gs_probe_ffma(float* out, int blocks, int iters, void* stream) {
  if (!out || blocks < 1 || iters < 1) return gs::set_error(GS_ERR_INVALID, "gs_probe_ffma: bad arguments");
  k_probe_ffma<<<blocks, 256, 0, gs::as_stream(stream)>>>(out, iters, 0.999999f, 1e-7f);
  return gs::check_launch("gs_probe_ffma");
}
