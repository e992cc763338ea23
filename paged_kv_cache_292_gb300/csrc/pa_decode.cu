// Host side of paged decode: the launch plan (heads per CTA, ranges, stage
// ring), the tensor maps of the pools, argument checks and the C entry
// points.  The kernel itself is in pa_decode_kernel.cuh.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <type_traits>

#include "../../include/pagedattn.h"
#include "pa_decode_kernel.cuh"
#include "pa_internal.h"
#include "pa_schedule.h"

namespace pa {

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

struct Plan {
  int Hg, HG, R, stages, q_slots, split;
  uint32_t row_bytes, pitch, q_bytes, stage_bytes, smem;
  uint32_t lines, box_rows, box_bytes;  // tensor-core paths (see DecodeParams)
  size_t ws_ml, ws_o, ws_partials, ws_counters, ws_total;
};

// Scratch layout: partial (m, l) and O at the start, then the merge tickets
// (num_seqs * num_kv_heads int32).  In a caller's buffer the tickets occupy
// its last bytes (rounded down to 256), so that buffers reused across batch
// shapes keep tickets and partials apart.
size_t workspace_layout(int num_seqs, int num_heads, int num_kv_heads, int head_size, int R,
                        Plan* pl, int num_queries = 1) {
  num_heads *= num_queries;  // partial rows are (query, head) pairs
  const size_t ml = align_up(sizeof(float) * (size_t)R * 2 * num_heads * 2, 256);
  const size_t o = align_up(sizeof(float) * (size_t)R * 2 * num_heads * head_size, 256);
  const size_t cnt = align_up(sizeof(int32_t) * (size_t)num_seqs * num_kv_heads, 256);
  if (pl) {
    pl->ws_ml = 0;
    pl->ws_o = ml;
    pl->ws_partials = ml + o;
    pl->ws_counters = cnt;
    pl->ws_total = ml + o + cnt;
  }
  return ml + o + cnt;
}

// KV heads one CTA stages per token row: the largest divisor of num_kv_heads
// that is at most `max_heads` (8 with one consumer warp per KV head, 4 with
// two) and keeps the row within 2 KiB, so three stages fit in shared memory.
int heads_per_cta(int num_kv_heads, int head_size, int elt, int max_heads = kMaxGroupHeads) {
  for (int h = max_heads; h > 1; --h)
    if (num_kv_heads % h == 0 && h * head_size * elt <= kMaxRowBytes) return h;
  return 1;
}

// Consumer warps per KV head: one 8-wide MMA tile of (query, head) columns
// per warp, so ceil(columns / 8) (at most 4: 32 columns).
int column_split(int group, int num_queries) { return (group * num_queries + 7) / 8; }

int default_ranges(const DeviceInfo& dev, int HG) {
  const int r = dev.sm_count / HG;
  return r < 1 ? 1 : r;
}

int gcd_int(int a, int b) {
  while (b != 0) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// elt: bytes of a pool element; q_elt: bytes of a query element (bf16 queries
// select the tensor-core consumers, whose stages are swizzled tensor boxes).
int make_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size, int elt,
              int num_ranges, const DeviceInfo& dev, Plan* pl, int num_queries = 1,
              int q_elt = 0, int block_size = 16) {
  if (q_elt == 0) q_elt = elt;
  const int G = num_heads / num_kv_heads;
  const bool mma = q_elt == 2;
  pl->split = column_split(G, num_queries);
  pl->Hg = heads_per_cta(num_kv_heads, head_size, elt, kMaxGroupHeads / pl->split);
  pl->HG = num_kv_heads / pl->Hg;
  pl->R = num_ranges > 0 ? num_ranges : default_ranges(dev, pl->HG);
  pl->row_bytes = (uint32_t)(pl->Hg * head_size * elt);
  pl->q_bytes = (uint32_t)(num_queries * pl->Hg * G * head_size * q_elt);
  pl->lines = pl->box_rows = pl->box_bytes = 0;
  if (mma) {
    if (pl->row_bytes % kLine != 0)
      return fail(PA_ERR_UNSUPPORTED,
                  "pa_decode: %d KV heads x %d dims make %u-byte rows, not whole 128-byte lines",
                  pl->Hg, head_size, pl->row_bytes);
    // A tensor copy moves box_rows = gcd(block_size, 16) rows (they share a
    // block) and must land on a 1 KiB boundary under the 128-byte swizzle, so
    // box_rows * lines is a multiple of 8: lines is a multiple of `step`.  An
    // odd multiple spreads consecutive rows over the most bank groups.
    const uint32_t chunks = pl->row_bytes / kLine;
    const int br = gcd_int(block_size, kTile);
    const uint32_t step = 8u / (uint32_t)gcd_int(br, 8);
    uint32_t lines = (chunks + step - 1) / step * step;
    if ((lines / step) % 2 == 0) lines += step;
    pl->lines = lines;
    pl->box_rows = (uint32_t)br;
    pl->box_bytes = (uint32_t)br * lines * kLine;
    pl->pitch = lines * kLine;
  } else {
    pl->pitch = pl->row_bytes + kRowSkew;
  }
  pl->stage_bytes = 2u * kTile * pl->pitch;
  pl->stages = 0;
  const int pref[][2] = {{6, 2}, {5, 2}, {4, 2}, {3, 2}, {3, 1}, {2, 2}, {2, 1}};
  for (auto& c : pref) {
    const Layout L = make_layout(c[0], c[1], pl->q_bytes, pl->stage_bytes, mma);
    if ((int)L.total <= dev.max_smem_optin) {
      pl->stages = c[0];
      pl->q_slots = c[1];
      pl->smem = L.total;
      break;
    }
  }
  if (pl->stages == 0)
    return fail(PA_ERR_UNSUPPORTED, "decode stages (%u bytes each) do not fit in %d bytes of shared memory",
                pl->stage_bytes, dev.max_smem_optin);
  // Consumers that take two tiles per pass (FP8 pools; bf16 with a KV head's
  // columns split over several warps) hold two stages at once: they need four
  // or more.  Their rows are at most 1 KiB, so every shape they accept has.
  const bool pairs = mma && (elt == 1 || pl->split >= 2);
  if (pairs && pl->stages < 4)
    return fail(PA_ERR_UNSUPPORTED, "decode: %d stages of %u bytes, four needed", pl->stages, pl->stage_bytes);
  workspace_layout(num_seqs, num_heads, num_kv_heads, head_size, pl->R, pl, num_queries);
  return PA_OK;
}

int validate(const void* out, const void* query, const void* k_cache, const void* v_cache,
             const int32_t* block_tables, const int32_t* context_lens, int num_seqs, int num_heads,
             int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq, float scale,
             int dtype, int num_physical_blocks, int num_ranges) {
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
    return fail(PA_ERR_INVALID_ARG, "pa_decode: null tensor pointer");
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return fail(PA_ERR_INVALID_ARG, "pa_decode: sizes must be positive");
  if (num_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "pa_decode: num_heads %d not a multiple of num_kv_heads %d",
                num_heads, num_kv_heads);
  if (num_heads / num_kv_heads > kMaxQueryGroup)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: query group %d > %d", num_heads / num_kv_heads,
                kMaxQueryGroup);
  if (head_size != 64 && head_size != 128)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: head_size %d (built: 64, 128)", head_size);
  if (block_size > 4096) return fail(PA_ERR_UNSUPPORTED, "pa_decode: block_size %d > 4096", block_size);
  if ((long long)max_blocks_per_seq * block_size > (1ll << 30))
    return fail(PA_ERR_INVALID_ARG, "pa_decode: max context %lld too large",
                (long long)max_blocks_per_seq * block_size);
  if (dtype != PA_F32 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_decode: dtype %d", dtype);
  if (!aligned(out, 16) || !aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return fail(PA_ERR_INVALID_ARG, "pa_decode: tensors must be 16-byte aligned");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "pa_decode: scale not finite");
  if (num_ranges > kMaxRanges)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: num_ranges %d > %d", num_ranges, kMaxRanges);
  if (num_physical_blocks < 0 || num_ranges < 0)
    return fail(PA_ERR_INVALID_ARG, "pa_decode: negative num_physical_blocks or num_ranges");
  return PA_OK;
}

// Launch with programmatic stream serialisation: the kernel may become
// resident while its predecessor on the stream finishes; it calls
// griddepcontrol.wait before touching anything that predecessor produces.
template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       const Params& prm) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

// The pools seen by the tensor copies: 4-D byte tensors (byte within a
// 128-byte chunk, chunk within a head group's row, head group, token row)
// with strides (1, 128, group row bytes, token row bytes).  A box is
// (128, lines, 1, box_rows); its lines past the group's row are outside the
// tensor, so they arrive zero-filled without touching memory.
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn encode_tiled_fn() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      return static_cast<EncodeTiledFn>(nullptr);
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// Encoded maps of the last few pools this thread decoded over.  A map is a
// pure function of the pool's address, extents, strides and box, which form
// the key, so a hit is exactly what a fresh encode would give; repeated
// steps over the same pools skip the driver call.
struct TensorMapCacheEntry {
  const void* k;
  const void* v;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  CUtensorMap tm_k, tm_v;
  bool used;
};
constexpr int kTensorMapCache = 4;
thread_local TensorMapCacheEntry g_tmap_cache[kTensorMapCache];
thread_local int g_tmap_next = 0;

int make_tensor_maps(DecodeParams* prm, const Plan& pl, int num_kv_heads, int head_size, int kv_elt,
                     int block_size, int num_physical_blocks) {
  const EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return fail(PA_ERR_CUDA, "pa_decode: the driver has no cuTensorMapEncodeTiled");
  // Unknown pool size: the row extent only has to cover every valid row, and
  // no pool that fits in device memory has 2^31 token rows of >= 128 bytes.
  const uint64_t rows =
      num_physical_blocks > 0 ? (uint64_t)num_physical_blocks * block_size : (1ull << 31);
  if (rows > (1ull << 31))
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: %llu token rows in the pool (at most 2^31)",
                (unsigned long long)rows);
  const cuuint64_t dims[4] = {kLine, pl.row_bytes / kLine, (cuuint64_t)pl.HG, rows};
  const cuuint64_t strides[3] = {kLine, pl.row_bytes,
                                 (cuuint64_t)num_kv_heads * head_size * kv_elt};
  const cuuint32_t box[4] = {kLine, pl.lines, 1u, pl.box_rows};
  const cuuint32_t estride[4] = {1u, 1u, 1u, 1u};
  for (int c = 0; c < kTensorMapCache; ++c) {
    const TensorMapCacheEntry& e = g_tmap_cache[c];
    if (e.used && e.k == prm->k_cache && e.v == prm->v_cache && memcmp(e.dims, dims, sizeof(dims)) == 0 &&
        memcmp(e.strides, strides, sizeof(strides)) == 0 && memcmp(e.box, box, sizeof(box)) == 0) {
      prm->tm_k = e.tm_k;
      prm->tm_v = e.tm_v;
      return PA_OK;
    }
  }
  for (int i = 0; i < 2; ++i) {
    const CUresult r = enc(i ? &prm->tm_v : &prm->tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                           const_cast<void*>(i ? prm->v_cache : prm->k_cache), dims, strides, box,
                           estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(PA_ERR_CUDA, "pa_decode: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  }
  TensorMapCacheEntry& e = g_tmap_cache[g_tmap_next];
  g_tmap_next = (g_tmap_next + 1) % kTensorMapCache;
  e.k = prm->k_cache;
  e.v = prm->v_cache;
  memcpy(e.dims, dims, sizeof(dims));
  memcpy(e.strides, strides, sizeof(strides));
  memcpy(e.box, box, sizeof(box));
  e.tm_k = prm->tm_k;
  e.tm_v = prm->tm_v;
  e.used = true;
  return PA_OK;
}

template <typename T, int D, int GMAX, int QMODE = 0, bool KV8 = false>
int launch_typed(const DecodeParams& prm, const Plan& pl, int dev, cudaStream_t stream) {
  // Devices whose shared-memory limit is already raised for this kernel
  // (setting it again is harmless, so concurrent first calls may both set it).
  constexpr int kTrackedDevices = 64;
  static std::atomic<bool> configured[kTrackedDevices];
  auto kern = pa_decode_kernel<T, D, GMAX, QMODE, KV8>;
  if (dev < 0 || dev >= kTrackedDevices || !configured[dev].load(std::memory_order_acquire)) {
    DeviceInfo info{};
    int rc = current_device_info(&info);
    if (rc != PA_OK) return rc;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, info.max_smem_optin);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(decode smem)");
    if (dev >= 0 && dev < kTrackedDevices) configured[dev].store(true, std::memory_order_release);
  }
  cudaError_t e =
      launch_pdl(kern, dim3(pl.R * pl.HG), dim3(32 * (pl.Hg * pl.split + kProducers)), pl.smem, stream, prm);
  if (e != cudaSuccess) return cuda_fail(e, "launch pa_decode_kernel");
  return PA_OK;
}

template <typename T, int D>
int launch_dtype(const DecodeParams& prm, const Plan& pl, int dev, cudaStream_t stream,
                 bool kv_fp8 = false) {
  if constexpr (sizeof(T) == 2) {
    if (kv_fp8) {
      if (prm.num_queries == 1) return launch_typed<T, D, 8, 0, true>(prm, pl, dev, stream);
      return prm.group * prm.num_queries <= 8 ? launch_typed<T, D, 8, 1, true>(prm, pl, dev, stream)
                                               : launch_typed<T, D, 8, 2, true>(prm, pl, dev, stream);
    }
    if (prm.num_queries > 1)  // (query, head) columns in one or two 8-wide MMA tiles
      return prm.group * prm.num_queries <= 8 ? launch_typed<T, D, 8, 1>(prm, pl, dev, stream)
                                               : launch_typed<T, D, 8, 2>(prm, pl, dev, stream);
    return launch_typed<T, D, 8>(prm, pl, dev, stream);  // the MMA consumer pads G to 8
  } else {
    const int G = prm.group;
    if (G <= 1) return launch_typed<T, D, 1>(prm, pl, dev, stream);
    if (G <= 2) return launch_typed<T, D, 2>(prm, pl, dev, stream);
    if (G <= 4) return launch_typed<T, D, 4>(prm, pl, dev, stream);
    return launch_typed<T, D, 8>(prm, pl, dev, stream);
  }
}

}  // namespace

// fixed_scratch: when set and `workspace` is NULL, the scratch comes from this
// provider (given the plan's byte count, it returns a device buffer that keeps
// earlier contents, or an error) instead of the library's growable buffer;
// its merge tickets are then cleared on `stream` right before the launch,
// after every check has passed.
int decode_impl_q(void* out, const void* query, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                  int num_queries, int num_heads, int num_kv_heads, int head_size, int block_size,
                  int max_blocks_per_seq, float scale, void* stream, int dtype,
                  int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                  int32_t* error_flag, bool kv_fp8 = false, float k_scale = 1.f,
                  float v_scale = 1.f, const void* k_new = nullptr, const void* v_new = nullptr,
                  ScratchProvider fixed_scratch = nullptr) {
  clear_error();
  if (k_new != nullptr || v_new != nullptr) {
    if (k_new == nullptr || v_new == nullptr)
      return fail(PA_ERR_INVALID_ARG, "pa_decode_append: k_new and v_new are both needed");
    if (dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_decode_append: bf16 queries and pools only");
    if (!aligned(k_new, 16) || !aligned(v_new, 16))
      return fail(PA_ERR_INVALID_ARG, "pa_decode_append: k_new / v_new not 16-byte aligned");
  }
  if (kv_fp8) {
    if (dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "pa_decode_fp8: query/out must be bf16");
    if (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale <= 0.f || v_scale <= 0.f)
      return fail(PA_ERR_INVALID_ARG, "pa_decode_fp8: scales must be finite and positive");
  }
  int rc = validate(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                    num_kv_heads, head_size, block_size, max_blocks_per_seq, scale, dtype,
                    num_physical_blocks, num_ranges);
  if (rc != PA_OK) return rc;
  if (num_queries < 1) return fail(PA_ERR_INVALID_ARG, "pa_decode_mq: num_queries %d < 1", num_queries);
  if (num_queries > 1 && dtype != PA_BF16)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_mq: several queries need bf16");
  if (num_queries > 1 && (num_heads / num_kv_heads) * num_queries > kMaxColumns)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_mq: group size x queries = %d > %d",
                (num_heads / num_kv_heads) * num_queries, kMaxColumns);
  DeviceInfo dev{};
  rc = current_device_info(&dev);
  if (rc != PA_OK) return rc;
  const int elt = dtype == PA_F32 ? 4 : 2;
  Plan pl{};
  rc = make_plan(num_seqs, num_heads, num_kv_heads, head_size, kv_fp8 ? 1 : elt, num_ranges, dev, &pl,
                 num_queries, elt, block_size);
  if (rc != PA_OK) return rc;
  int32_t* counters = nullptr;
  const bool clear_tickets = workspace == nullptr && fixed_scratch != nullptr;
  if (clear_tickets) {
    rc = fixed_scratch(pl.ws_total, &workspace);
    if (rc != PA_OK) return rc;
    workspace_bytes = pl.ws_total;
  }
  if (workspace == nullptr) {
    rc = library_workspace(pl.ws_partials, &workspace);
    if (rc != PA_OK) return rc;
    rc = library_counters(pl.ws_counters, &counters);
    if (rc != PA_OK) return rc;
  } else {
    if (workspace_bytes < pl.ws_total)
      return fail(PA_ERR_WORKSPACE, "pa_decode: workspace of %zu bytes, %zu needed", workspace_bytes,
                  pl.ws_total);
    if (!aligned(workspace, 256)) return fail(PA_ERR_INVALID_ARG, "pa_decode: workspace not 256-byte aligned");
    const size_t cnt_bytes = sizeof(int32_t) * (size_t)num_seqs * num_kv_heads;
    counters = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) +
                                          ((workspace_bytes - cnt_bytes) & ~(size_t)255));
  }
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  DecodeParams prm{};
  prm.out = out;
  prm.q = query;
  prm.k_cache = k_cache;
  prm.v_cache = v_cache;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.counters = counters;
  prm.part_ml = reinterpret_cast<float*>(ws + pl.ws_ml);
  prm.part_o = reinterpret_cast<float*>(ws + pl.ws_o);
  prm.error_flag = error_flag;
  prm.num_seqs = num_seqs;
  prm.num_heads = num_heads;
  prm.num_kv_heads = num_kv_heads;
  prm.group = num_heads / num_kv_heads;
  prm.block_size = block_size;
  prm.max_blocks_per_seq = max_blocks_per_seq;
  prm.heads_per_cta = pl.Hg;
  prm.num_head_groups = pl.HG;
  prm.num_ranges = pl.R;
  prm.num_physical_blocks = num_physical_blocks;
  prm.stages = pl.stages;
  prm.num_queries = num_queries;
  prm.split = pl.split;
  prm.q_slots = pl.q_slots;
  prm.row_bytes = pl.row_bytes;
  prm.pitch = pl.pitch;
  prm.q_bytes = pl.q_bytes;
  prm.stage_bytes = pl.stage_bytes;
  prm.lines = pl.lines;
  prm.box_rows = pl.box_rows;
  prm.box_bytes = pl.box_bytes;
  if (dtype == PA_BF16) {
    rc = make_tensor_maps(&prm, pl, num_kv_heads, head_size, kv_fp8 ? 1 : 2, block_size,
                          num_physical_blocks);
    if (rc != PA_OK) return rc;
  }
  prm.scale_log2 = (float)((double)scale * (double)k_scale * 1.4426950408889634);
  prm.v_scale = v_scale;
  prm.k_scale = k_scale;
  prm.k_new = k_new;
  prm.v_new = v_new;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clear_tickets) {
    const cudaError_t e =
        cudaMemsetAsync(counters, 0, sizeof(int32_t) * (size_t)num_seqs * num_kv_heads, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(merge tickets)");
  }
  take_wait_test(&prm.stall_tile, &prm.wait_limit_ns);
  if (k_new != nullptr && pl.split >= 2) {
    // Several consumer warps per KV head: the rows are written by their own
    // kernel, chained ahead of the decode, which then only reads them.
    rc = append_rows_impl(k_new, v_new, block_tables, context_lens, const_cast<void*>(k_cache),
                          const_cast<void*>(v_cache), num_seqs, num_queries, num_kv_heads, head_size,
                          block_size, max_blocks_per_seq, num_physical_blocks, stream, error_flag,
                          kv_fp8, k_scale, v_scale);
    if (rc != PA_OK) return rc;
    prm.k_new = prm.v_new = nullptr;
  }
  if (dtype == PA_BF16) {
    return head_size == 64 ? launch_dtype<__nv_bfloat16, 64>(prm, pl, dev.device, st, kv_fp8)
                           : launch_dtype<__nv_bfloat16, 128>(prm, pl, dev.device, st, kv_fp8);
  }
  return head_size == 64 ? launch_dtype<float, 64>(prm, pl, dev.device, st)
                         : launch_dtype<float, 128>(prm, pl, dev.device, st);
}

int decode_impl(void* out, const void* query, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                int num_heads, int num_kv_heads, int head_size, int block_size,
                int max_blocks_per_seq, float scale, void* stream, int dtype,
                int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                int32_t* error_flag) {
  return decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                       num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                       stream, dtype, num_physical_blocks, workspace, workspace_bytes, num_ranges,
                       error_flag);
}

size_t decode_workspace_size_q(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                               int num_ranges, int num_queries) {
  if (num_queries < 1) return 0;
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || num_ranges < 0 ||
      num_heads % num_kv_heads != 0)
    return 0;
  int R = num_ranges;
  if (R == 0) {
    DeviceInfo dev{};
    if (current_device_info(&dev) != PA_OK) return 0;
    // The head grouping depends on the element size; size for bf16, whose
    // larger groups leave more ranges per head group.
    const int split = column_split(num_heads / num_kv_heads, num_queries);
    R = default_ranges(dev, num_kv_heads / heads_per_cta(num_kv_heads, head_size, 2, kMaxGroupHeads / split));
  }
  return workspace_layout(num_seqs, num_heads, num_kv_heads, head_size, R, nullptr, num_queries);
}

size_t decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                             int num_ranges) {
  return decode_workspace_size_q(num_seqs, num_heads, num_kv_heads, head_size, num_ranges, 1);
}

}  // namespace pa

extern "C" int pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                         int num_heads, int num_kv_heads, int head_size, int block_size,
                         int max_blocks_per_seq, float scale, void* stream, int dtype) {
  return pa::decode_impl(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                         num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                         stream, dtype, 0, nullptr, 0, 0, nullptr);
}

extern "C" int pa_decode_ws(void* out, const void* query, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_size,
                            int block_size, int max_blocks_per_seq, float scale, void* stream,
                            int dtype, void* workspace, size_t workspace_bytes) {
  if (workspace == nullptr) {
    pa::clear_error();
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_ws: null workspace");
  }
  return pa::decode_impl(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                         num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                         stream, dtype, 0, workspace, workspace_bytes, 0, nullptr);
}

extern "C" int pa_decode_ex(void* out, const void* query, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int num_heads, int num_kv_heads, int head_size,
                            int block_size, int max_blocks_per_seq, float scale, void* stream,
                            int dtype, int num_physical_blocks, void* workspace,
                            size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  return pa::decode_impl(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                         num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                         stream, dtype, num_physical_blocks, workspace, workspace_bytes, num_ranges,
                         error_flag);
}

extern "C" int pa_decode_append(void* out, const void* query, const void* k_new, const void* v_new,
                                void* k_cache, void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, int num_seqs, int num_heads,
                                int num_kv_heads, int head_size, int block_size,
                                int max_blocks_per_seq, float scale, void* stream, int dtype,
                                int num_physical_blocks, void* workspace, size_t workspace_bytes,
                                int num_ranges, int32_t* error_flag) {
  if (k_new == nullptr || v_new == nullptr) {
    pa::clear_error();
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_append: null k_new / v_new");
  }
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                           stream, dtype, num_physical_blocks, workspace, workspace_bytes, num_ranges,
                           error_flag, false, 1.f, 1.f, k_new, v_new);
}

extern "C" int pa_decode_fp8_append(void* out, const void* query, const void* k_new, const void* v_new,
                                    void* k_cache, void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, int num_seqs, int num_heads,
                                    int num_kv_heads, int head_size, int block_size,
                                    int max_blocks_per_seq, float scale, float k_scale, float v_scale,
                                    void* stream, int num_physical_blocks, void* workspace,
                                    size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  if (k_new == nullptr || v_new == nullptr) {
    pa::clear_error();
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_fp8_append: null k_new / v_new");
  }
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                           stream, PA_BF16, num_physical_blocks, workspace, workspace_bytes, num_ranges,
                           error_flag, true, k_scale, v_scale, k_new, v_new);
}

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                           int head_size, int num_ranges) {
  return pa::decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, num_ranges);
}

extern "C" int pa_decode_mq(void* out, const void* query, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int num_seqs, int num_queries, int num_heads, int num_kv_heads,
                            int head_size, int block_size, int max_blocks_per_seq, float scale,
                            void* stream, int dtype, int num_physical_blocks, void* workspace,
                            size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           num_queries, num_heads, num_kv_heads, head_size, block_size,
                           max_blocks_per_seq, scale, stream, dtype, num_physical_blocks, workspace,
                           workspace_bytes, num_ranges, error_flag);
}

extern "C" int pa_decode_mq_append(void* out, const void* query, const void* k_new, const void* v_new,
                                   void* k_cache, void* v_cache, const int32_t* block_tables,
                                   const int32_t* context_lens, int num_seqs, int num_queries,
                                   int num_heads, int num_kv_heads, int head_size, int block_size,
                                   int max_blocks_per_seq, float scale, void* stream, int dtype,
                                   int num_physical_blocks, void* workspace, size_t workspace_bytes,
                                   int num_ranges, int32_t* error_flag) {
  if (k_new == nullptr || v_new == nullptr) {
    pa::clear_error();
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_mq_append: null k_new / v_new");
  }
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           num_queries, num_heads, num_kv_heads, head_size, block_size,
                           max_blocks_per_seq, scale, stream, dtype, num_physical_blocks, workspace,
                           workspace_bytes, num_ranges, error_flag, false, 1.f, 1.f, k_new, v_new);
}

extern "C" size_t pa_decode_mq_workspace_size(int num_seqs, int num_queries, int num_heads,
                                              int num_kv_heads, int head_size, int num_ranges) {
  return pa::decode_workspace_size_q(num_seqs, num_heads, num_kv_heads, head_size, num_ranges,
                                     num_queries);
}

extern "C" int pa_decode_fp8(void* out, const void* query, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int num_seqs, int num_heads, int num_kv_heads, int head_size,
                             int block_size, int max_blocks_per_seq, float scale, float k_scale,
                             float v_scale, void* stream, int num_physical_blocks, void* workspace,
                             size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, 1,
                           num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                           stream, PA_BF16, num_physical_blocks, workspace, workspace_bytes,
                           num_ranges, error_flag, true, k_scale, v_scale);
}

extern "C" int pa_decode_fp8_mq(void* out, const void* query, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                                int num_queries, int num_heads, int num_kv_heads, int head_size,
                                int block_size, int max_blocks_per_seq, float scale, float k_scale,
                                float v_scale, void* stream, int num_physical_blocks, void* workspace,
                                size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           num_queries, num_heads, num_kv_heads, head_size, block_size,
                           max_blocks_per_seq, scale, stream, PA_BF16, num_physical_blocks, workspace,
                           workspace_bytes, num_ranges, error_flag, true, k_scale, v_scale);
}

extern "C" int pa_decode_fp8_mq_append(void* out, const void* query, const void* k_new, const void* v_new,
                                       void* k_cache, void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, int num_seqs, int num_queries,
                                       int num_heads, int num_kv_heads, int head_size, int block_size,
                                       int max_blocks_per_seq, float scale, float k_scale, float v_scale,
                                       void* stream, int num_physical_blocks, void* workspace,
                                       size_t workspace_bytes, int num_ranges, int32_t* error_flag) {
  if (k_new == nullptr || v_new == nullptr) {
    pa::clear_error();
    return pa::fail(PA_ERR_INVALID_ARG, "pa_decode_fp8_mq_append: null k_new / v_new");
  }
  return pa::decode_impl_q(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           num_queries, num_heads, num_kv_heads, head_size, block_size,
                           max_blocks_per_seq, scale, stream, PA_BF16, num_physical_blocks, workspace,
                           workspace_bytes, num_ranges, error_flag, true, k_scale, v_scale, k_new, v_new);
}
