// pa_decode_static: paged decode that allocates nothing.
//
// Some callers cannot call cudaMalloc at the point where they decode: a
// serving engine whose own allocator has already reserved nearly all device
// memory (a fresh cudaMalloc then fails or fragments its pool), or a latency
// path that cannot afford cudaMalloc/cudaFree's implicit device
// synchronisation.  pa_decode allocates its scratch on first use and
// pa_decode_ws needs the caller to provide some; this entry point instead uses
// a fixed scratch array compiled into the library.  The caller still passes
// every input and output buffer.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library holds PA_STATIC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, not a device address; the
// device address is fetched once per device with cudaGetSymbolAddress, with
// that device current, on the first call made on that device.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_SCRATCH_BYTES];

namespace pa {

int decode_impl_q(void* out, const void* query, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                  int num_queries, int num_heads, int num_kv_heads, int head_size, int block_size,
                  int max_blocks_per_seq, float scale, void* stream, int dtype,
                  int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                  int32_t* error_flag, bool kv_fp8, float k_scale, float v_scale, const void* k_new,
                  const void* v_new, ScratchProvider fixed_scratch);

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
void* g_static_ptr[kMaxDevices] = {nullptr};

// The scratch array as the decode's fixed scratch: rejects batches that need
// more than it holds, and returns its device address on the current device
// (looked up once per device, with that device current).
int static_scratch(size_t bytes, void** ptr) {
  if (bytes > (size_t)PA_STATIC_SCRATCH_BYTES)
    return fail(PA_ERR_WORKSPACE,
                "pa_decode_static: this batch needs %zu bytes of scratch, more than the %zu "
                "compiled in (use pa_decode or pa_decode_ws)",
                bytes, (size_t)PA_STATIC_SCRATCH_BYTES);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return PA_OK;
}
}  // namespace

}  // namespace pa

// The arguments are checked exactly as pa_decode checks them (same codes, and
// nothing is queued on the stream for a rejected call); the scratch array then
// stands in for the library's buffer, and its merge tickets are cleared on the
// caller's stream just before the kernel.
extern "C" int pa_decode_static(void* out, const void* query, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_size, int block_size,
                                int max_blocks_per_seq, float scale, void* stream, int dtype) {
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                           stream, dtype, 0, nullptr, 0, 0, nullptr, false, 1.f, 1.f, nullptr,
                           nullptr, pa::static_scratch);
}
