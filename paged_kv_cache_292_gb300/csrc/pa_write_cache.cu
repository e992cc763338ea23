// Cache write ("reshape_and_cache"): scatter one step's new K/V rows into the
// paged pool through slot_mapping.
//
// Follows section 2 item 4 of "vLLM three-process architecture and the
// PagedAttention kernel" (the new token joins its sequence's current physical
// block) and section 4 item 3, which calls the kernel's access pattern a
// gather-scatter: decode gathers through the block table, this kernel scatters
// through the slot of each new token.
//
// In the [block, slot, kv_head, dim] pool one token's K (or V) for all KV heads
// is a single contiguous row of num_kv_heads * head_size elements at row index
// `slot` (block * block_size + offset).  So the scatter is a byte copy of whole
// rows with 16-byte vector accesses; one CTA per token copies its K and V rows.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(128) pa_write_cache_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int num_tokens, int row_vecs, long long num_slots,
    int32_t* error_flag) {
  griddep_wait();               // new rows may come from the kernel just before
  griddep_launch_dependents();  // a following decode may get resident; it waits for us
  for (int i = blockIdx.x; i < num_tokens; i += gridDim.x) {
    const long long slot = slot_mapping[i];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (threadIdx.x == 0) report(error_flag, PA_DEVERR_SLOT);
      continue;
    }
    const uint4* ks = k_new + (size_t)i * row_vecs;
    const uint4* vs = v_new + (size_t)i * row_vecs;
    uint4* kd = k_cache + (size_t)slot * row_vecs;
    uint4* vd = v_cache + (size_t)slot * row_vecs;
    for (int j = threadIdx.x; j < row_vecs; j += blockDim.x) {
      const uint4 kv = __ldg(ks + j);
      const uint4 vv = __ldg(vs + j);
      kd[j] = kv;
      vd[j] = vv;
    }
  }
}

int write_cache_impl(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                     void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                     int head_size, int block_size, int num_physical_blocks, void* stream,
                     int dtype, int32_t* error_flag) {
  clear_error();
  if (!k_cache || !v_cache || (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)))
    return fail(PA_ERR_INVALID_ARG, "pa_write_cache: null tensor pointer");
  if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      num_physical_blocks <= 0)
    return fail(PA_ERR_INVALID_ARG, "pa_write_cache: sizes must be positive");
  if (dtype != PA_F32 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "pa_write_cache: dtype %d", dtype);
  const long long row_bytes = (long long)num_kv_heads * head_size * (dtype == PA_F32 ? 4 : 2);
  if (row_bytes % 16 != 0)
    return fail(PA_ERR_UNSUPPORTED, "pa_write_cache: row of %lld bytes is not a multiple of 16",
                row_bytes);
  if (row_bytes / 16 > (1 << 24)) return fail(PA_ERR_UNSUPPORTED, "pa_write_cache: row too long");
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return fail(PA_ERR_INVALID_ARG, "pa_write_cache: tensors must be 16-byte aligned");
  if (num_tokens == 0) return PA_OK;
  const long long num_slots = (long long)num_physical_blocks * block_size;
  const int grid = num_tokens < 65535 ? num_tokens : 65535;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, pa_write_cache_kernel, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      slot_mapping, static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_tokens,
      static_cast<int>(row_bytes / 16), num_slots, error_flag);
  if (e != cudaSuccess) return cuda_fail(e, "launch pa_write_cache_kernel");
  return PA_OK;
}

// The new rows of a multi-query appending call, for shapes whose decode does
// not write them itself: token i of sequence s (row s * Q + i of k_new /
// v_new) sits at position c - Q + i of its sequence, so its slot comes from
// the block table.  Tokens before the sequence's start are skipped; lengths
// outside [0, max_blocks_per_seq * block_size] are clamped as the decode
// clamps them, and a failed block-id check (num_physical_blocks > 0) leaves
// the token unwritten and sets PA_DEVERR_BLOCK_ID.  One CTA per token.
// KV8: the pools are FP8 (E4M3); each bf16 element x becomes the code of the
// fp32 quotient x / scale, saturating, with the FP8 cache write's own
// conversion, four codes per 32-bit store.  row_units counts 16-byte units of
// a bf16 row (8 elements each).
template <bool KV8>
__global__ void __launch_bounds__(128) pa_append_rows_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, const int32_t* __restrict__ block_tables,
    const int32_t* __restrict__ context_lens, void* __restrict__ k_cache, void* __restrict__ v_cache,
    int num_seqs, int num_queries, int block_size, int max_blocks_per_seq, int row_units,
    int num_physical_blocks, float k_scale, float v_scale, int32_t* error_flag) {
  griddep_wait();
  griddep_launch_dependents();
  const long long n = (long long)num_seqs * num_queries;
  for (long long i = blockIdx.x; i < n; i += gridDim.x) {
    const int s = (int)(i / num_queries), qi = (int)(i % num_queries);
    const int cmax = max_blocks_per_seq * block_size;
    const int c = min(max(context_lens[s], 0), cmax);
    const int pos = c - num_queries + qi;
    if (pos < 0) continue;
    const int blk = block_tables[(size_t)s * max_blocks_per_seq + pos / block_size];
    if (num_physical_blocks > 0 && (blk < 0 || blk >= num_physical_blocks)) {
      if (threadIdx.x == 0) report(error_flag, PA_DEVERR_BLOCK_ID);
      continue;
    }
    const size_t slot = (size_t)blk * block_size + pos % block_size;
    const uint4* ks = k_new + (size_t)i * row_units;
    const uint4* vs = v_new + (size_t)i * row_units;
    for (int j = threadIdx.x; j < row_units; j += blockDim.x) {
      const uint4 kv = __ldg(ks + j);
      const uint4 vv = __ldg(vs + j);
      if constexpr (KV8) {
        // 8 bf16 elements -> 8 codes (two 32-bit words) per pool.
        const uint4 src[2] = {kv, vv};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float sc = h ? v_scale : k_scale;
          const uint32_t w[4] = {src[h].x, src[h].y, src[h].z, src[h].w};
          uint32_t code[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(bf16_lo(w[2 * e]) / sc, bf16_hi(w[2 * e]) / sc), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(bf16_lo(w[2 * e + 1]) / sc, bf16_hi(w[2 * e + 1]) / sc), __NV_SATFINITE,
                __NV_E4M3);
            code[e] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
          }
          uint2* dst = static_cast<uint2*>(h ? v_cache : k_cache) + slot * row_units + j;
          *dst = make_uint2(code[0], code[1]);
        }
      } else {
        static_cast<uint4*>(k_cache)[slot * row_units + j] = kv;
        static_cast<uint4*>(v_cache)[slot * row_units + j] = vv;
      }
    }
  }
}

// Launches pa_append_rows_kernel (programmatic dependent launch, like the
// cache write).  Arguments are validated by the caller (bf16 rows of
// num_kv_heads * head_size elements, 16-byte aligned).
int append_rows_impl(const void* k_new, const void* v_new, const int32_t* block_tables,
                     const int32_t* context_lens, void* k_cache, void* v_cache, int num_seqs,
                     int num_queries, int num_kv_heads, int head_size, int block_size,
                     int max_blocks_per_seq, int num_physical_blocks, void* stream, int32_t* error_flag,
                     bool kv_fp8, float k_scale, float v_scale) {
  const long long n = (long long)num_seqs * num_queries;
  if (n <= 0) return PA_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n < 65535 ? n : 65535));
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int units = num_kv_heads * head_size * 2 / 16;
  const cudaError_t e =
      kv_fp8 ? cudaLaunchKernelEx(&cfg, pa_append_rows_kernel<true>, static_cast<const uint4*>(k_new),
                                  static_cast<const uint4*>(v_new), block_tables, context_lens, k_cache, v_cache,
                                  num_seqs, num_queries, block_size, max_blocks_per_seq, units,
                                  num_physical_blocks, k_scale, v_scale, error_flag)
             : cudaLaunchKernelEx(&cfg, pa_append_rows_kernel<false>, static_cast<const uint4*>(k_new),
                                  static_cast<const uint4*>(v_new), block_tables, context_lens, k_cache, v_cache,
                                  num_seqs, num_queries, block_size, max_blocks_per_seq, units,
                                  num_physical_blocks, 1.f, 1.f, error_flag);
  if (e != cudaSuccess) return cuda_fail(e, "launch pa_append_rows_kernel");
  return PA_OK;
}

}  // namespace pa

extern "C" int pa_write_cache(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                              void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                              int head_size, int block_size, int num_physical_blocks,
                              void* stream, int dtype) {
  return pa::write_cache_impl(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens,
                              num_kv_heads, head_size, block_size, num_physical_blocks, stream,
                              dtype, nullptr);
}

extern "C" int pa_write_cache_ex(const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                 int num_tokens, int num_kv_heads, int head_size, int block_size,
                                 int num_physical_blocks, void* stream, int dtype,
                                 int32_t* error_flag) {
  return pa::write_cache_impl(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens,
                              num_kv_heads, head_size, block_size, num_physical_blocks, stream,
                              dtype, error_flag);
}

// ---------------------------------------------------------------------------
// Copy-on-write support: whole-block copies inside both pools.
// ---------------------------------------------------------------------------
namespace pa {

__global__ void __launch_bounds__(256) pa_copy_blocks_kernel(uint4* __restrict__ k_cache,
                                                             uint4* __restrict__ v_cache,
                                                             const int32_t* __restrict__ pairs,
                                                             int num_pairs, int block_vecs,
                                                             int num_blocks) {
  griddep_wait();
  for (int i = blockIdx.x; i < num_pairs; i += gridDim.x) {
    const int src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) continue;
    const size_t so = (size_t)src * block_vecs, d = (size_t)dst * block_vecs;
    for (int j = threadIdx.x; j < block_vecs; j += blockDim.x) {
      k_cache[d + j] = k_cache[so + j];
      v_cache[d + j] = v_cache[so + j];
    }
  }
}

}  // namespace pa

extern "C" int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                              int num_kv_heads, int head_size, int block_size,
                              int num_physical_blocks, void* stream, int dtype) {
  pa::clear_error();
  if (!k_cache || !v_cache || (num_pairs > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: null pointer");
  if (num_pairs < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_physical_blocks <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: sizes must be positive");
  if (dtype != PA_F32 && dtype != PA_BF16) return pa::fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: dtype %d", dtype);
  const long long bytes = (long long)block_size * num_kv_heads * head_size * (dtype == PA_F32 ? 4 : 2);
  if (bytes % 16 != 0 || bytes / 16 > (1ll << 30))
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_copy_blocks: block of %lld bytes", bytes);
  if (!pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16) || !pa::aligned(pairs, 4))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_copy_blocks: misaligned pointer");
  if (num_pairs == 0) return PA_OK;
  const int grid = num_pairs < 65535 ? num_pairs : 65535;
  pa::pa_copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), pairs, num_pairs,
      static_cast<int>(bytes / 16), num_physical_blocks);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return pa::cuda_fail(e, "launch pa_copy_blocks_kernel");
  return PA_OK;
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) pool: quantising cache write.
// ---------------------------------------------------------------------------
namespace pa {

template <typename T>
__global__ void __launch_bounds__(128) pa_write_cache_fp8_kernel(
    const T* __restrict__ k_new, const T* __restrict__ v_new, const int64_t* __restrict__ slot_mapping,
    uint32_t* __restrict__ k_cache, uint32_t* __restrict__ v_cache, int num_tokens, int row_elems,
    long long num_slots, float k_scale, float v_scale, int32_t* error_flag) {
  griddep_wait();
  griddep_launch_dependents();
  const int quads = row_elems / 4;
  for (int i = blockIdx.x; i < num_tokens; i += gridDim.x) {
    const long long slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (threadIdx.x == 0) report(error_flag, PA_DEVERR_SLOT);
      continue;
    }
    for (int j = threadIdx.x; j < 2 * quads; j += blockDim.x) {
      const bool is_v = j >= quads;
      const int qj = is_v ? j - quads : j;
      const T* src = (is_v ? v_new : k_new) + (size_t)i * row_elems + 4 * qj;
      const float sc = is_v ? v_scale : k_scale;
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = static_cast<float>(src[e]) / sc;  // IEEE division
      const __nv_fp8x2_storage_t lo =
          __nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3);
      const __nv_fp8x2_storage_t hi =
          __nv_cvt_float2_to_fp8x2(make_float2(x[2], x[3]), __NV_SATFINITE, __NV_E4M3);
      uint32_t* dst = (is_v ? v_cache : k_cache) + (size_t)slot * quads + qj;
      *dst = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
  }
}

}  // namespace pa

extern "C" int pa_write_cache_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                  void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                                  int head_size, int block_size, int num_physical_blocks,
                                  float k_scale, float v_scale, void* stream, int src_dtype,
                                  int32_t* error_flag) {
  pa::clear_error();
  if (!k_cache || !v_cache || (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_write_cache_fp8: null tensor pointer");
  if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_physical_blocks <= 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_write_cache_fp8: sizes must be positive");
  if (src_dtype != PA_F32 && src_dtype != PA_BF16)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_write_cache_fp8: source dtype %d", src_dtype);
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale > 3.0e38f || v_scale > 3.0e38f)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_write_cache_fp8: scales must be finite and positive");
  const long long row_elems = (long long)num_kv_heads * head_size;
  if (row_elems % 16 != 0 || row_elems > (1 << 24))
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_write_cache_fp8: row of %lld elements", row_elems);
  if (!pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16) || !pa::aligned(k_new, 16) ||
      !pa::aligned(v_new, 16) || !pa::aligned(slot_mapping, 8))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_write_cache_fp8: misaligned pointer");
  if (num_tokens == 0) return PA_OK;
  const long long num_slots = (long long)num_physical_blocks * block_size;
  const int grid = num_tokens < 65535 ? num_tokens : 65535;
  // Programmatic dependent launch, as for pa_write_cache: the kernel may become
  // resident while the one before it finishes and waits for it in-kernel.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (src_dtype == PA_BF16)
    e = cudaLaunchKernelEx(&cfg, pa::pa_write_cache_fp8_kernel<__nv_bfloat16>,
                           static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
                           slot_mapping, static_cast<uint32_t*>(k_cache), static_cast<uint32_t*>(v_cache),
                           num_tokens, (int)row_elems, num_slots, k_scale, v_scale, error_flag);
  else
    e = cudaLaunchKernelEx(&cfg, pa::pa_write_cache_fp8_kernel<float>, static_cast<const float*>(k_new),
                           static_cast<const float*>(v_new), slot_mapping, static_cast<uint32_t*>(k_cache),
                           static_cast<uint32_t*>(v_cache), num_tokens, (int)row_elems, num_slots, k_scale,
                           v_scale, error_flag);
  if (e != cudaSuccess) return pa::cuda_fail(e, "launch pa_write_cache_fp8_kernel");
  return PA_OK;
}
