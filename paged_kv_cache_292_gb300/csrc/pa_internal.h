// Host-side helpers shared by the library's translation units (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// Record a message for pa_last_error() and return `code`.
int fail(int code, const char* fmt, ...);
// Record a CUDA failure (with its runtime message) and return PA_ERR_CUDA.
int cuda_fail(cudaError_t err, const char* what);
// Clear the calling thread's message.
void clear_error();

struct DeviceInfo {
  int device;
  int sm_count;
  int max_smem_optin;  // bytes of dynamic shared memory one CTA may opt into
};

// Properties of the current device (cached per device; no synchronisation).
int current_device_info(DeviceInfo* info);

// Library-owned scratch for the current device, grown to at least `bytes`.
// Growing frees the old buffer (cudaFree synchronises the device).
int library_workspace(size_t bytes, void** ptr);

// Library-owned, zero-filled merge-ticket buffer for the current device, grown
// to at least `bytes` (zero-filled again when it grows).
int library_counters(size_t bytes, int32_t** ptr);

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace pa
