// Host-side plumbing: per-thread error messages, cached device properties and
// the library-owned decode scratch.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

namespace pa {

namespace {
thread_local char g_message[512] = {0};
// pa_test_stall_copy: consumed by the next decode launch on this thread.
thread_local long long g_stall_tile = -1;
thread_local unsigned int g_stall_limit_us = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices] = {false};
void* g_ws_ptr[kMaxDevices] = {nullptr};
size_t g_ws_bytes[kMaxDevices] = {0};
void* g_cnt_ptr[kMaxDevices] = {nullptr};
size_t g_cnt_bytes[kMaxDevices] = {0};
}  // namespace

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_message, sizeof(g_message), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
}

void clear_error() { g_message[0] = '\0'; }

int current_device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_info_valid[dev]) {
    DeviceInfo d{};
    d.device = dev;
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(sm count)");
    e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem optin)");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major * 10 + minor != 103)
      return fail(PA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only",
                  dev, major, minor);
    g_info[dev] = d;
    g_info_valid[dev] = true;
  }
  *info = g_info[dev];
  return PA_OK;
}

int library_workspace(size_t bytes, void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_ws_bytes[dev] < bytes) {
    if (g_ws_ptr[dev] != nullptr) {
      e = cudaFree(g_ws_ptr[dev]);
      g_ws_ptr[dev] = nullptr;
      g_ws_bytes[dev] = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree(workspace)");
    }
    const size_t want = align_up(bytes < (1u << 20) ? (1u << 20) : bytes, 1u << 20);
    e = cudaMalloc(&g_ws_ptr[dev], want);
    if (e != cudaSuccess) {
      g_ws_ptr[dev] = nullptr;
      return cuda_fail(e, "cudaMalloc(workspace)");
    }
    g_ws_bytes[dev] = want;
  }
  *ptr = g_ws_ptr[dev];
  return PA_OK;
}

int library_counters(size_t bytes, int32_t** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_cnt_bytes[dev] < bytes) {
    if (g_cnt_ptr[dev] != nullptr) {
      e = cudaFree(g_cnt_ptr[dev]);
      g_cnt_ptr[dev] = nullptr;
      g_cnt_bytes[dev] = 0;
      if (e != cudaSuccess) return cuda_fail(e, "cudaFree(tickets)");
    }
    const size_t want = align_up(bytes < 65536 ? 65536 : bytes, 65536);
    void* p = nullptr;
    e = cudaMalloc(&p, want);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(tickets)");
    // Merge tickets start at zero; every completed decode leaves them zero.
    e = cudaMemset(p, 0, want);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
      cudaFree(p);
      return cuda_fail(e, "cudaMemset(tickets)");
    }
    g_cnt_ptr[dev] = p;
    g_cnt_bytes[dev] = want;
  }
  *ptr = static_cast<int32_t*>(g_cnt_ptr[dev]);
  return PA_OK;
}

void take_wait_test(long long* stall_tile, unsigned long long* wait_limit_ns) {
  *stall_tile = g_stall_tile;
  *wait_limit_ns = g_stall_limit_us ? 1000ull * g_stall_limit_us : 2000000000ull;
  g_stall_tile = -1;
  g_stall_limit_us = 0;
}

}  // namespace pa

extern "C" int pa_test_stall_copy(long long tile, unsigned int wait_limit_us) {
  pa::clear_error();
  if (tile < -1) return pa::fail(PA_ERR_INVALID_ARG, "pa_test_stall_copy: tile %lld < -1", tile);
  pa::g_stall_tile = tile;
  pa::g_stall_limit_us = tile < 0 ? 0u : wait_limit_us;
  return PA_OK;
}

extern "C" const char* pa_last_error(void) { return pa::g_message; }

extern "C" int pa_version(void) { return 100; }
