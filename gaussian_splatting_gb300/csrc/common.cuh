// Shared helpers of the libgs.so kernels: status plumbing, launch checks, small vector math.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gs.h"

namespace gs {

constexpr int kTile = 16;            // pixels per tile edge
constexpr int kTilePixels = kTile * kTile;

// Host-side error reporting (per host thread); defined in api.cu.
gs_status set_error(gs_status s, const char* fmt, ...);
gs_status check_launch(const char* what);
int64_t wait_limit();
int take_drop_publish();
int num_sms();
// cudaFuncSetAttribute(fn, MaxDynamicSharedMemorySize, bytes) for the current device, made once
// per device (and kernel) -- the attribute is per device, so a second device gets its own call
cudaError_t max_dynamic_smem(const void* fn, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Camera as the kernels see it (by value in the launch parameters).
struct Cam {
  float R[9];
  float t[3];
  float fx, fy, cx, cy, znear;
  int W, H, Tx, Ty;
};

inline Cam make_cam(const gs_camera& c) {
  Cam k;
  for (int i = 0; i < 9; ++i) k.R[i] = c.R[i];
  for (int i = 0; i < 3; ++i) k.t[i] = c.t[i];
  k.fx = c.fx; k.fy = c.fy; k.cx = c.cx; k.cy = c.cy; k.znear = c.znear;
  k.W = c.width; k.H = c.height;
  k.Tx = (c.width + kTile - 1) / kTile;
  k.Ty = (c.height + kTile - 1) / kTile;
  return k;
}

inline gs_status check_camera(const gs_camera* cam) {
  if (!cam) return set_error(GS_ERR_INVALID, "camera is NULL");
  if (cam->width <= 0 || cam->height <= 0 || cam->width > 32768 || cam->height > 32768)
    return set_error(GS_ERR_INVALID, "bad image size %d x %d", cam->width, cam->height);
  if (!(cam->fx > 0.f) || !(cam->fy > 0.f)) return set_error(GS_ERR_INVALID, "focal lengths must be > 0");
  return GS_OK;
}

// Status bits written to device memory by kernels.
constexpr int64_t kStatusCapacity = 1;
constexpr int64_t kStatusTimeout = 2;

}  // namespace gs

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float4 ld4(const float* base, int64_t i) {
  return reinterpret_cast<const float4*>(base)[i];
}
__device__ __forceinline__ float4 ldg4(const float* base, int64_t i) {
  return __ldg(reinterpret_cast<const float4*>(base) + i);
}
__device__ __forceinline__ void st4(float* base, int64_t i, float4 v) {
  reinterpret_cast<float4*>(base)[i] = v;
}

// exp2 on the special-function unit (PTX ex2.approx: relative error ~2^-22).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte vector atomic add to global memory (sm_90+).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Acquire loads / release stores for flags other CTAs poll (grid barriers).
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
