/*
 * pagedattn.h - C ABI of the GB300 (sm_103a) paged decode-attention library.
 *
 * The operation is the PagedAttention decode step described in "vLLM
 * three-process architecture and the PagedAttention kernel" (devpress.csdn.net),
 * section 3 "PagedAttention 内核原理：从概念到 CUDA 实现":
 *   3.1 "输入是什么": query[num_seqs, num_heads, head_size],
 *       block_tables[num_seqs, max_blocks_per_seq],
 *       k_cache / v_cache[num_physical_blocks, block_size, num_kv_heads, head_size];
 *   3.2 "内核执行流程（简化版）": for each sequence, read its block table (step 1),
 *       derive the number of logical blocks from its valid length (step 2),
 *       gather K/V from the scattered physical blocks (step 3), run standard
 *       attention with the step's query (step 4), write the output (step 5).
 * Section 2 "工作流程拆解", item 4, appends each new token's K/V into the
 * sequence's current physical block: pa_write_cache.
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is DEVICE memory owned by the caller, dense and
 *     row-major in the shape given.  The library never frees or keeps it.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream and never synchronise the host.
 *   - The return value is PA_OK (0) or a negative PA_ERR_* code; on error
 *     nothing was launched and pa_last_error() describes the cause.
 *   - `dtype` is PA_F32 or PA_BF16 and applies to query, out, the pools and
 *     the new K/V rows alike.  Arithmetic is fp32 in every case.
 *   - Query head h reads KV head h / (num_heads / num_kv_heads).
 *   - context_lens[s] counts every valid token of sequence s, including the
 *     current step's (written by pa_write_cache first).  Token t of sequence s
 *     is row t % block_size of physical block block_tables[s][t / block_size].
 *     Table entries at or past ceil(context_lens[s] / block_size) are never
 *     read.  Pool rows no valid token occupies never affect the result; the
 *     bf16 and FP8 decode paths do read the unused rows of a sequence's last,
 *     partly filled block (they copy whole runs of rows), so those rows must
 *     lie in the pool, but their contents (even NaN) do not matter.
 *     context_lens[s] == 0 gives an all-zero output row.
 *   - Device-detected input faults (a block id outside [0, num_physical_blocks),
 *     a context length beyond max_blocks_per_seq * block_size or negative, a
 *     slot outside the pool) are reported by OR-ing PA_DEVERR_* bits into the
 *     optional device word `error_flag`; the offending row is skipped (its
 *     content is then unspecified) instead of being read or written.
 *   - Kernels are launched with programmatic stream serialisation: a kernel
 *     may become resident while the one before it on the stream finishes, but
 *     it reads and writes nothing until that kernel has completed
 *     (griddepcontrol.wait).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define PA_OK 0
#define PA_ERR_INVALID_ARG (-1) /* null pointer, bad size, misaligned pointer */
#define PA_ERR_UNSUPPORTED (-2) /* valid but not built: head_size, group size, dtype */
#define PA_ERR_CUDA (-3)        /* a CUDA runtime call failed (message kept) */
#define PA_ERR_WORKSPACE (-4)   /* caller workspace smaller than required */

/* Element types. */
#define PA_F32 0
#define PA_BF16 1
#define PA_FP8_E4M3 2 /* pool element only: 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448 */

/* Bits OR-ed into the optional device error word. */
#define PA_DEVERR_BLOCK_ID 1    /* block id outside [0, num_physical_blocks) */
#define PA_DEVERR_CONTEXT_LEN 2 /* context length < 0 or > max_blocks_per_seq*block_size (clamped) */
#define PA_DEVERR_SLOT 4        /* slot_mapping entry >= num_physical_blocks*block_size (skipped) */
#define PA_DEVERR_TIMEOUT 8     /* a pipeline wait exceeded its limit; the kernel returned early */

/*
 * pa_decode - paged decode attention, one query token per sequence.
 *
 *   out[s, h, :] = sum_t softmax_t(scale * <query[s, h, :], K_s[t, h/G, :]>) V_s[t, h/G, :]
 *
 * out          [num_seqs, num_heads, head_size], dtype            (written)
 * query        [num_seqs, num_heads, head_size], dtype
 * k_cache      [num_physical_blocks, block_size, num_kv_heads, head_size], dtype
 * v_cache      same shape as k_cache
 * block_tables [num_seqs, max_blocks_per_seq] int32
 * context_lens [num_seqs] int32
 * Requirements: num_heads % num_kv_heads == 0 and num_heads / num_kv_heads <= 8;
 * head_size 64 or 128; block_size in [1, 4096]; query, out and both pools
 * 16-byte aligned; for bf16, fewer than 2^31 token rows in the pool
 * (num_physical_blocks * block_size) else PA_ERR_UNSUPPORTED.
 * bf16 pools are read through TMA tensor maps built on the host for each call
 * (cuTensorMapEncodeTiled, taken from the driver; PA_ERR_CUDA if the driver
 * lacks it); block sizes that are multiples of 8 stream fastest.
 * The batch's tiles of 16 tokens are split into equal ranges, one CTA each.
 * A sequence cut by range boundaries leaves partial softmax statistics per
 * range; the last CTA to finish one of its KV heads merges them by
 * log-sum-exp in a second pass over the partials.  The scratch for that comes
 * from a per-device buffer the library allocates (zero-filled) on first use
 * and grows when a larger batch needs it (cudaMalloc, which synchronises the
 * device; use pa_decode_ws to supply the scratch and never allocate).  That
 * buffer is shared by every call on the device: calls that may run at the
 * same time on different streams must use pa_decode_ws with scratch of their
 * own.
 */
int pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
              int num_heads, int num_kv_heads, int head_size, int block_size,
              int max_blocks_per_seq, float scale, void* stream, int dtype);

/*
 * pa_decode_workspace_size - bytes of scratch pa_decode_ws needs on the
 * current device for this batch shape (num_ranges as in pa_decode_ex; 0 =
 * the default of one range per SM).  Returns 0 for invalid sizes.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                int num_ranges);

/*
 * pa_decode_ws - pa_decode with caller-owned scratch (device memory of at
 * least pa_decode_workspace_size(...) bytes, 256-byte aligned).  Never
 * allocates.  The scratch must be zero-filled before its first use; every
 * call that completes leaves it zero-filled again, so it can be reused by the
 * next call on the same stream.  Two calls that overlap in time must not
 * share it.  After a call that reported PA_DEVERR_TIMEOUT, zero it again.
 */
int pa_decode_ws(void* out, const void* query, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                 int num_heads, int num_kv_heads, int head_size, int block_size,
                 int max_blocks_per_seq, float scale, void* stream, int dtype, void* workspace,
                 size_t workspace_bytes);

/*
 * pa_decode_ex - the general form behind pa_decode and pa_decode_ws.
 *
 * num_physical_blocks  > 0: every block id read from block_tables is checked
 *                      against it on the device (PA_DEVERR_BLOCK_ID); 0: unchecked.
 * workspace            NULL: library-owned scratch (may allocate, see pa_decode).
 * num_ranges           0: one token range per SM (the default).  > 0: split the
 *                      flattened batch into exactly this many ranges (1 = a
 *                      single CTA walks every sequence in one pass).
 * error_flag           optional device int32 that receives PA_DEVERR_* bits.
 */
int pa_decode_ex(void* out, const void* query, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                 int num_heads, int num_kv_heads, int head_size, int block_size,
                 int max_blocks_per_seq, float scale, void* stream, int dtype,
                 int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                 int32_t* error_flag);

/*
 * pa_decode_append - one decode step with its cache write fused in: for every
 * sequence s with context_lens[s] >= 1, the K/V of its newest token (position
 * context_lens[s] - 1) are k_new[s] / v_new[s]; the call stores them into the
 * pool at that position (block_tables[s][(c-1) / block_size], row
 * (c-1) % block_size) and returns the same `out` as pa_write_cache of those
 * rows followed by pa_decode_ex.  One launch instead of two: the decode
 * itself puts the new rows into its staged tile and into the pool.
 * k_new, v_new  [num_seqs, num_kv_heads, head_size], 16-byte aligned
 * The newest token's block must not be shared with another sequence of the
 * batch (copy-on-write first, as pa_bm_append arranges).  dtype PA_BF16 only
 * (PA_ERR_UNSUPPORTED otherwise; FP8 pools: pa_decode_fp8_append).  Other arguments as in pa_decode_ex; a
 * failed block-id check (num_physical_blocks > 0) leaves that token unwritten.
 */
int pa_decode_append(void* out, const void* query, const void* k_new, const void* v_new,
                     void* k_cache, void* v_cache, const int32_t* block_tables,
                     const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                     int head_size, int block_size, int max_blocks_per_seq, float scale,
                     void* stream, int dtype, int num_physical_blocks, void* workspace,
                     size_t workspace_bytes, int num_ranges, int32_t* error_flag);

/*
 * pa_decode_mq - several query tokens per sequence over the paged cache, with
 * a causal mask: the chunked-prefill / speculative-decoding-verification step
 * (named by the vLLM book preface's reader questions and the is96 essay's
 * feature list) built on the same gather as pa_decode.
 *
 *   out[s, i, h, :] = attention of query[s, i, h, :] over the keys/values at
 *                     positions 0 .. context_lens[s] - num_queries + i
 *
 * query, out  [num_seqs, num_queries, num_heads, head_size]
 * The num_queries newest tokens of every sequence must already be in the pool
 * (pa_write_cache) and counted in context_lens.  A query whose position is
 * negative (context shorter than num_queries) gets a zero row.
 * Requires dtype PA_BF16 and (num_heads / num_kv_heads) * num_queries <= 32;
 * num_queries == 1 is plain decode.  Other arguments as in pa_decode_ex; the
 * scratch size comes from pa_decode_mq_workspace_size (workspace NULL: the
 * library's own, allocated on first use).
 */
int pa_decode_mq(void* out, const void* query, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                 int num_queries, int num_heads, int num_kv_heads, int head_size, int block_size,
                 int max_blocks_per_seq, float scale, void* stream, int dtype,
                 int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                 int32_t* error_flag);

/* Scratch bytes pa_decode_mq needs (0 for invalid sizes). */
size_t pa_decode_mq_workspace_size(int num_seqs, int num_queries, int num_heads, int num_kv_heads,
                                   int head_size, int num_ranges);

/*
 * pa_decode_mq_append - pa_decode_mq with the step's cache write fused in: for
 * every sequence s with context c = context_lens[s], the K/V of its query
 * token i (position c - num_queries + i) are k_new[s * num_queries + i] /
 * v_new[s * num_queries + i]; the call stores each token whose position is
 * >= 0 into the pool (block_tables[s][pos / block_size], row
 * pos % block_size) and returns the same `out` as pa_write_cache of those
 * rows followed by pa_decode_mq.  One launch instead of two when
 * (num_heads / num_kv_heads) * num_queries <= 8; above that (two to four
 * consumer warps per KV head) the call launches a row-writing kernel and then the
 * decode on `stream`, chained by programmatic dependent launch.
 * k_new, v_new  [num_seqs * num_queries, num_kv_heads, head_size], bf16,
 *               16-byte aligned
 * The blocks of the new tokens must not be shared with another sequence of
 * the batch.  dtype PA_BF16 only (PA_ERR_UNSUPPORTED otherwise).  Other
 * arguments, scratch size and limits as in pa_decode_mq; a failed block-id
 * check (num_physical_blocks > 0) leaves that token unwritten.
 */
int pa_decode_mq_append(void* out, const void* query, const void* k_new, const void* v_new,
                        void* k_cache, void* v_cache, const int32_t* block_tables,
                        const int32_t* context_lens, int num_seqs, int num_queries, int num_heads,
                        int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                        float scale, void* stream, int dtype, int num_physical_blocks,
                        void* workspace, size_t workspace_bytes, int num_ranges,
                        int32_t* error_flag);

/*
 * pa_write_cache - scatter one step's new K/V rows into the paged pool
 * (the "reshape_and_cache" step).  For every token i with slot_mapping[i] >= 0:
 *   k_cache[slot / block_size, slot % block_size, :, :] = k_new[i, :, :]  (bit copy)
 * and the same for V.  Negative slots are padding and are skipped; slots at
 * or beyond num_physical_blocks * block_size are skipped and reported.
 * Duplicate slots within one call leave either row (unspecified which).
 * k_new, v_new  [num_tokens, num_kv_heads, head_size], dtype, 16-byte aligned
 * slot_mapping  [num_tokens] int64
 * k_cache, v_cache as in pa_decode (written in place).
 */
int pa_write_cache(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                   void* k_cache, void* v_cache, int num_tokens, int num_kv_heads, int head_size,
                   int block_size, int num_physical_blocks, void* stream, int dtype);

/* pa_write_cache_ex - pa_write_cache with an optional device error word. */
int pa_write_cache_ex(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                      void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                      int head_size, int block_size, int num_physical_blocks, void* stream,
                      int dtype, int32_t* error_flag);

/*
 * pa_decode_static - pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot call cudaMalloc when they decode, e.g. a serving engine whose
 * own allocator has already reserved nearly all device memory, or a latency
 * path that cannot afford cudaMalloc's implicit device synchronisation.
 * Arguments, layouts and results are those of pa_decode.  Instead of
 * allocating scratch it uses an array of PA_STATIC_SCRATCH_BYTES compiled
 * into the library: every GPU that loads the library holds that memory until
 * the process exits.  Nothing is allocated or freed by this call.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Arguments are checked as pa_decode checks them, with the same return
 *     codes; a rejected call queues nothing on `stream`.
 *   - All calls share the one array, which keeps the previous call's
 *     contents; each accepted call clears the part that must start at zero
 *     (cudaMemsetAsync on `stream`) right before its kernel.  Calls that
 *     overlap in time on the GPU (different streams, no ordering) race on
 *     the array.
 *   - Batches whose scratch exceeds PA_STATIC_SCRATCH_BYTES are rejected with
 *     PA_ERR_WORKSPACE before anything is queued (the scratch is at most
 *     pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, 0)
 *     bytes: about 5 MB for 64 sequences of 32 query / 8 KV heads of 128).
 */
#define PA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
int pa_decode_static(void* out, const void* query, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_size, int block_size,
                     int max_blocks_per_seq, float scale, void* stream, int dtype);

/*
 * FP8 KV pool.  The pages list quantisation among vLLM's features but give no
 * format; this library's reading: the pool holds E4M3 codes with one float
 * scale per pool (k_scale, v_scale), a code c standing for e4m3(c) * scale.
 *
 * pa_write_cache_fp8 - pa_write_cache into FP8 pools: each new element x
 * becomes the E4M3 code nearest to x / scale (the quotient in float32, ties to
 * even, saturating at +-448).  k_new/v_new are PA_BF16 or PA_F32 (src_dtype);
 * k_cache/v_cache are uint8 [num_physical_blocks, block_size, num_kv_heads,
 * head_size].  error_flag as in pa_write_cache_ex (optional).
 *
 * pa_decode_fp8 - pa_decode_ex over FP8 pools (one query per sequence; several:
 * pa_decode_fp8_mq), query and out bf16: scores use
 * k = e4m3(code) * k_scale and values v = e4m3(code) * v_scale.  Each token
 * moves half the bytes of a bf16 pool.  Scratch as pa_decode_workspace_size.
 * The query is rounded to f16 on the way into the tensor cores (exact for
 * |q| in [2^-14, 65504]).  head_size 64 with an odd num_kv_heads is
 * PA_ERR_UNSUPPORTED (a KV-head group's FP8 row must be whole 128-byte lines).
 */
int pa_write_cache_fp8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                       void* k_cache, void* v_cache, int num_tokens, int num_kv_heads, int head_size,
                       int block_size, int num_physical_blocks, float k_scale, float v_scale,
                       void* stream, int src_dtype, int32_t* error_flag);
int pa_decode_fp8(void* out, const void* query, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                  int num_heads, int num_kv_heads, int head_size, int block_size,
                  int max_blocks_per_seq, float scale, float k_scale, float v_scale, void* stream,
                  int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                  int32_t* error_flag);

/*
 * pa_decode_fp8_append - pa_decode_append over FP8 pools: the newest token's
 * bf16 K/V (k_new/v_new [num_seqs, num_kv_heads, head_size]) are quantised
 * as pa_write_cache_fp8 does (bit-identical codes) and written into the pools
 * by the decode launch itself; out equals pa_write_cache_fp8 followed by
 * pa_decode_fp8.  Scales, layouts and limits as in pa_decode_fp8.
 */
int pa_decode_fp8_append(void* out, const void* query, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                         int head_size, int block_size, int max_blocks_per_seq, float scale,
                         float k_scale, float v_scale, void* stream, int num_physical_blocks,
                         void* workspace, size_t workspace_bytes, int num_ranges, int32_t* error_flag);

/*
 * pa_decode_fp8_mq - pa_decode_mq over FP8 pools: several causal query tokens
 * per sequence (chunked prefill, speculative-decoding verification) reading
 * the quantised cache.  Keys and values are e4m3(code) * k_scale and
 * e4m3(code) * v_scale as in pa_decode_fp8; query and out are bf16
 * [num_seqs, num_queries, num_heads, head_size]; query i of sequence s sees
 * positions 0 .. context_lens[s] - num_queries + i.  Requires
 * (num_heads / num_kv_heads) * num_queries <= 32.  Scratch size:
 * pa_decode_mq_workspace_size.  Other arguments and limits as in
 * pa_decode_fp8 and pa_decode_mq.
 *
 * pa_decode_fp8_mq_append - the same with the step's quantising cache write
 * fused in: k_new / v_new [num_seqs * num_queries, num_kv_heads, head_size]
 * bf16 (row s * num_queries + i: position context_lens[s] - num_queries + i)
 * are quantised as pa_write_cache_fp8 does (bit-identical codes) and stored
 * into the pools; tokens at negative positions are skipped.  Up to 8
 * (query, head) columns per KV head the decode launch itself writes them;
 * above that a row-writing kernel is chained ahead of the decode.  out equals
 * pa_write_cache_fp8 of those rows followed by pa_decode_fp8_mq.
 */
int pa_decode_fp8_mq(void* out, const void* query, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                     int num_queries, int num_heads, int num_kv_heads, int head_size, int block_size,
                     int max_blocks_per_seq, float scale, float k_scale, float v_scale, void* stream,
                     int num_physical_blocks, void* workspace, size_t workspace_bytes, int num_ranges,
                     int32_t* error_flag);
int pa_decode_fp8_mq_append(void* out, const void* query, const void* k_new, const void* v_new,
                            void* k_cache, void* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, int num_seqs, int num_queries, int num_heads,
                            int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                            float scale, float k_scale, float v_scale, void* stream,
                            int num_physical_blocks, void* workspace, size_t workspace_bytes,
                            int num_ranges, int32_t* error_flag);

/*
 * pa_test_stall_copy - test hook for the decode kernel's bounded waits; the
 * pages have no counterpart.  Every wait of the decode pipeline (a consumer
 * waiting for a stage's copies, the copy engine's issuer waiting for a free
 * stage) gives up after a time limit, sets PA_DEVERR_TIMEOUT in error_flag and
 * ends the kernel early, so that a copy that never lands cannot hang the GPU.
 * This hook lets a test reach that path without any fault: the next decode
 * call on the calling thread that launches its kernel (pa_decode*, any
 * variant) withholds every copy of flattened tile `tile` (the batch's tiles of
 * 16 tokens, sequence after sequence, counted from 0) and bounds every wait by
 * wait_limit_us microseconds (0: the default of 2 s).  The stage meant for
 * that tile is never filled, the waits on it run out, and the kernel returns
 * after letting the copies it had started land (again within the limit).
 * That call's output is unspecified, and its scratch (pa_decode_ws) must be
 * zero-filled again before reuse.  The setting is used by one launch and then
 * cleared; tile = -1 clears it.  Returns PA_OK, or PA_ERR_INVALID_ARG for
 * tile < -1.
 */
int pa_test_stall_copy(long long tile, unsigned int wait_limit_us);

/* Message for the calling thread's last non-zero return ("" if none). */
const char* pa_last_error(void);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
