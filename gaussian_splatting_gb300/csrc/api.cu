// Host-side plumbing shared by every entry point: per-thread error messages, launch
// checks, test hooks for the bounded device waits.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"

namespace {
thread_local std::string g_last_error;
std::atomic<int64_t> g_wait_limit{int64_t(1) << 22};
std::atomic<int> g_drop_publish{0};
}  // namespace

namespace gs {

gs_status set_error(gs_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gs_status check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(GS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return GS_OK;
}

int64_t wait_limit() { return g_wait_limit.load(); }

int take_drop_publish() { return g_drop_publish.exchange(0); }

cudaError_t max_dynamic_smem(const void* fn, int bytes) {
  // the attribute belongs to a device: remembered per device (and kernel, and size), so
  // that the driver call is made once per device rather than on every launch
  constexpr int kMaxDev = 64, kMaxEntries = 32;
  struct Entry {
    const void* fn;
    int bytes;
  };
  static std::mutex mu;
  static Entry done[kMaxDev][kMaxEntries];
  static int used[kMaxDev] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used[dev]; ++i)
    if (done[dev][i].fn == fn && done[dev][i].bytes >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) {
    for (int i = 0; i < used[dev]; ++i)
      if (done[dev][i].fn == fn) {
        done[dev][i].bytes = bytes;
        return e;
      }
    if (used[dev] < kMaxEntries) done[dev][used[dev]++] = Entry{fn, bytes};
  }
  return e;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

}  // namespace gs

extern "C" {

const char* gs_last_error(void) { return g_last_error.c_str(); }

int gs_version(void) { return 1; }

void gs_debug_set_wait_limit(int64_t iterations) {
  g_wait_limit.store(iterations < 1 ? (int64_t(1) << 22) : iterations);
}

void gs_debug_drop_publish(int mode) { g_drop_publish.store(mode == 1 || mode == 2 ? mode : 0); }

}  // extern "C"
