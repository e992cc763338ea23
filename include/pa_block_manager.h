/*
 * pa_block_manager.h - host-side paged KV block manager (C ABI).
 *
 * Implements the allocator the PagedAttention pages put beside the kernel:
 * "vLLM three-process architecture and the PagedAttention kernel"
 * (devpress.csdn.net), section 1.2 "引擎进程" (KVCacheManager): physical KV
 * memory split into fixed-size blocks, a global pool of free blocks, blocks
 * handed to a sequence on request, a logical-to-physical block table per
 * sequence, and reference counts with copy-on-write so that sequences (beam
 * search) can share blocks; section 2 item 4: a new token gets a new block
 * when the current one is full.  The vLLM book preface ("前言：走进 LLM 推理引擎
 * 的心脏", section "从 OS 到 GPU") adds that blocks are mapped on demand and
 * freed blocks are reused at once; the course page (aiflowlearn.net, "前缀缓存")
 * describes requests reusing the KV blocks of a common prefix.
 *
 * Everything here is host memory and host code; the manager never touches
 * the device.  It produces what the device kernels consume: per-token slots
 * for pa_write_cache, block tables and context lengths for pa_decode, and
 * (src, dst) block pairs for pa_copy_blocks when a shared block must be
 * copied before it is written.
 *
 * Conventions: sequences are numbered 0..max_seqs-1; a sequence slot is
 * empty until tokens are appended to it (or it is forked into).  Functions
 * return PA_OK (0) or a negative PA_ERR_* code from pagedattn.h and leave the
 * manager unchanged on error; pa_last_error() has the message.  A manager is
 * not thread-safe: one caller thread at a time.
 */
#ifndef PA_BLOCK_MANAGER_H
#define PA_BLOCK_MANAGER_H

#include <stdint.h>

#include "pagedattn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ERR_NO_BLOCKS (-5) /* the free pool cannot supply the blocks needed */

typedef struct pa_block_manager pa_block_manager;

/* A manager for a pool of num_blocks blocks of block_size tokens.  NULL on
 * invalid sizes (pa_last_error says why). */
pa_block_manager* pa_bm_create(int num_blocks, int block_size, int max_seqs, int max_blocks_per_seq);
void pa_bm_destroy(pa_block_manager* bm);

int pa_bm_num_free_blocks(const pa_block_manager* bm);
int pa_bm_context_len(const pa_block_manager* bm, int seq); /* <0 on a bad seq */
int pa_bm_ref_count(const pa_block_manager* bm, int block);  /* <0 on a bad block */

/*
 * pa_bm_append - make room for `num_tokens` more tokens at the end of `seq`
 * and return their slots (block * block_size + offset) in slots_out.
 * Blocks come from the free pool on demand.  If the sequence's last block is
 * shared (reference count > 1) and the first new token lands in it, the
 * sequence first gets a private copy: a fresh block replaces it in the table
 * and the pair (old, new) is written to copies_out[0..1] with *num_copies = 1
 * (else 0); the caller copies that block on the device (pa_copy_blocks)
 * before writing the new tokens.  copies_out needs room for 2 ints.
 * PA_ERR_NO_BLOCKS if the pool is short; PA_ERR_INVALID_ARG if the sequence
 * would exceed max_blocks_per_seq.
 */
int pa_bm_append(pa_block_manager* bm, int seq, int num_tokens, int64_t* slots_out,
                 int32_t* copies_out, int* num_copies);

/*
 * pa_bm_append_batch - pa_bm_append for several sequences in one call (one
 * decode step of a batch): sequence seqs[i] gets counts[i] tokens; their
 * slots are written back to back into slots_out (sum(counts) entries) and any
 * copy-on-write pairs into copies_out (room for 2 * num_seqs ints), with
 * their number in *num_copies.  On error the sequences before the failing one
 * keep their new tokens; *num_done tells how many sequences were served.
 */
int pa_bm_append_batch(pa_block_manager* bm, int num_seqs, const int32_t* seqs,
                       const int32_t* counts, int64_t* slots_out, int32_t* copies_out,
                       int* num_copies, int* num_done);

/* pa_bm_fork - `child` (empty) shares every block of `parent`: same table,
 * reference counts raised (beam search). */
int pa_bm_fork(pa_block_manager* bm, int parent, int child);

/* pa_bm_share_prefix - `seq` (empty) starts with the first `num_tokens` tokens
 * of `donor`, which must be a whole number of blocks: the donor's blocks are
 * shared, not copied (prefix caching). */
int pa_bm_share_prefix(pa_block_manager* bm, int seq, int donor, int num_tokens);

/* pa_bm_free - drop a sequence; blocks whose count reaches zero go back to
 * the front of the free pool (reused first). */
int pa_bm_free(pa_block_manager* bm, int seq);

/* pa_bm_export - write the block tables (int32 [max_seqs][max_blocks_per_seq],
 * -1 past each sequence's blocks) and context lengths (int32 [max_seqs], 0 for
 * empty slots) into host buffers, ready to copy to the device for pa_decode. */
int pa_bm_export(const pa_block_manager* bm, int32_t* block_tables, int32_t* context_lens);

/*
 * pa_copy_blocks - device copy of whole KV blocks (both pools) for
 * copy-on-write: for i < num_pairs, block pairs[2i+1] of k_cache and v_cache
 * becomes a bit copy of block pairs[2i].  pairs is DEVICE int32
 * [num_pairs][2]; pools as in pa_decode.  Asynchronous on `stream`.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                   int num_kv_heads, int head_size, int block_size, int num_physical_blocks,
                   void* stream, int dtype);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H */
