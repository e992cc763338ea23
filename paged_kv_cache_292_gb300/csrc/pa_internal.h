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

// Writes the new rows of a multi-query appending call into the pools (token
// i of sequence s at position context_lens[s] - num_queries + i), as its own
// kernel launch on `stream`.  bf16 rows; kv_fp8: quantised into FP8 pools as
// pa_write_cache_fp8 does (k_scale, v_scale).  The caller validates the
// arguments.
int append_rows_impl(const void* k_new, const void* v_new, const int32_t* block_tables,
                     const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                     int num_queries, int num_kv_heads, int head_size, int block_size,
                     int max_blocks_per_seq, int num_physical_blocks, void* stream, int32_t* error_flag,
                     bool kv_fp8 = false, float k_scale = 1.f, float v_scale = 1.f);

// The settings of pa_test_stall_copy for the decode launch about to be made on
// this thread (then cleared): the tile whose copies are withheld (-1: none)
// and the bound of every pipeline wait in nanoseconds.
void take_wait_test(long long* stall_tile, unsigned long long* wait_limit_ns);

// Supplies fixed (never allocated) decode scratch of at least `bytes` on the
// current device, or returns an error code (PA_ERR_WORKSPACE when too small).
typedef int (*ScratchProvider)(size_t bytes, void** ptr);

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace pa
