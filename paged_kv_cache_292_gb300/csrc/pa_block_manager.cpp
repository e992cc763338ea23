// Host-side paged KV block manager: free pool, on-demand allocation, block
// tables, reference counts with copy-on-write, prefix sharing.  See
// include/pa_block_manager.h for the contract and the passages it follows.
#include "../../include/pa_block_manager.h"

#include <deque>
#include <new>
#include <vector>

#include "pa_internal.h"

struct pa_block_manager {
  int num_blocks = 0, block_size = 0, max_seqs = 0, max_blocks = 0;
  std::vector<int> ref;                 // reference count per physical block
  std::deque<int> free_pool;            // front = next block handed out
  std::vector<std::vector<int>> table;  // logical -> physical, per sequence
  std::vector<int> len;                 // tokens per sequence
};

namespace {

bool bad_seq(const pa_block_manager* bm, int seq) {
  return bm == nullptr || seq < 0 || seq >= bm->max_seqs;
}

int take_block(pa_block_manager* bm) {
  const int b = bm->free_pool.front();
  bm->free_pool.pop_front();
  bm->ref[b] = 1;
  return b;
}

void drop_block(pa_block_manager* bm, int b) {
  if (--bm->ref[b] == 0) bm->free_pool.push_front(b);  // freed blocks are reused first
}

}  // namespace

extern "C" pa_block_manager* pa_bm_create(int num_blocks, int block_size, int max_seqs,
                                          int max_blocks_per_seq) {
  pa::clear_error();
  if (num_blocks <= 0 || block_size <= 0 || max_seqs <= 0 || max_blocks_per_seq <= 0) {
    pa::fail(PA_ERR_INVALID_ARG, "pa_bm_create: sizes must be positive");
    return nullptr;
  }
  pa_block_manager* bm = new (std::nothrow) pa_block_manager();
  if (bm == nullptr) {
    pa::fail(PA_ERR_INVALID_ARG, "pa_bm_create: out of host memory");
    return nullptr;
  }
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->max_seqs = max_seqs;
  bm->max_blocks = max_blocks_per_seq;
  bm->ref.assign(num_blocks, 0);
  for (int b = 0; b < num_blocks; ++b) bm->free_pool.push_back(b);
  bm->table.assign(max_seqs, std::vector<int>());
  bm->len.assign(max_seqs, 0);
  return bm;
}

extern "C" void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

extern "C" int pa_bm_num_free_blocks(const pa_block_manager* bm) {
  return bm ? static_cast<int>(bm->free_pool.size()) : PA_ERR_INVALID_ARG;
}

extern "C" int pa_bm_context_len(const pa_block_manager* bm, int seq) {
  return bad_seq(bm, seq) ? PA_ERR_INVALID_ARG : bm->len[seq];
}

extern "C" int pa_bm_ref_count(const pa_block_manager* bm, int block) {
  if (bm == nullptr || block < 0 || block >= bm->num_blocks) return PA_ERR_INVALID_ARG;
  return bm->ref[block];
}

extern "C" int pa_bm_append(pa_block_manager* bm, int seq, int num_tokens, int64_t* slots_out,
                            int32_t* copies_out, int* num_copies) {
  pa::clear_error();
  if (bad_seq(bm, seq) || num_tokens < 0 || (num_tokens > 0 && slots_out == nullptr) ||
      copies_out == nullptr || num_copies == nullptr)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append: bad sequence or null output");
  *num_copies = 0;
  const int bs = bm->block_size;
  std::vector<int>& tab = bm->table[seq];
  const long long cur = bm->len[seq];
  const long long want = cur + num_tokens;
  const long long need_blocks = (want + bs - 1) / bs;
  if (need_blocks > bm->max_blocks)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append: sequence %d would need %lld blocks > %d", seq,
                    need_blocks, bm->max_blocks);
  // The first new token goes into the current last block if it has room; a
  // shared last block must then be copied first.
  const bool cow = num_tokens > 0 && cur % bs != 0 && bm->ref[tab.back()] > 1;
  const long long fresh = need_blocks - static_cast<long long>(tab.size()) + (cow ? 1 : 0);
  if (fresh > static_cast<long long>(bm->free_pool.size()))
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_append: %lld blocks needed, %zu free", fresh,
                    bm->free_pool.size());
  if (cow) {
    const int old = tab.back();
    const int copy = take_block(bm);
    drop_block(bm, old);
    tab.back() = copy;
    copies_out[0] = old;
    copies_out[1] = copy;
    *num_copies = 1;
  }
  while (static_cast<long long>(tab.size()) < need_blocks) tab.push_back(take_block(bm));
  for (int i = 0; i < num_tokens; ++i) {
    const long long t = cur + i;
    slots_out[i] = static_cast<int64_t>(tab[t / bs]) * bs + t % bs;
  }
  bm->len[seq] = static_cast<int>(want);
  return PA_OK;
}

extern "C" int pa_bm_append_batch(pa_block_manager* bm, int num_seqs, const int32_t* seqs,
                                  const int32_t* counts, int64_t* slots_out, int32_t* copies_out,
                                  int* num_copies, int* num_done) {
  pa::clear_error();
  if (bm == nullptr || num_seqs < 0 || (num_seqs > 0 && (!seqs || !counts || !slots_out)) ||
      !copies_out || !num_copies || !num_done)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_batch: null argument");
  *num_copies = 0;
  *num_done = 0;
  int64_t* slot = slots_out;
  for (int i = 0; i < num_seqs; ++i) {
    int nc = 0;
    const int rc = pa_bm_append(bm, seqs[i], counts[i], slot, copies_out + 2 * *num_copies, &nc);
    if (rc != PA_OK) return rc;
    *num_copies += nc;
    slot += counts[i];
    *num_done = i + 1;
  }
  return PA_OK;
}

extern "C" int pa_bm_fork(pa_block_manager* bm, int parent, int child) {
  pa::clear_error();
  if (bad_seq(bm, parent) || bad_seq(bm, child) || parent == child)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_fork: bad sequence index");
  if (bm->len[child] != 0 || !bm->table[child].empty())
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_fork: child %d is not empty", child);
  bm->table[child] = bm->table[parent];
  for (int b : bm->table[child]) ++bm->ref[b];
  bm->len[child] = bm->len[parent];
  return PA_OK;
}

extern "C" int pa_bm_share_prefix(pa_block_manager* bm, int seq, int donor, int num_tokens) {
  pa::clear_error();
  if (bad_seq(bm, seq) || bad_seq(bm, donor) || seq == donor || num_tokens < 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_share_prefix: bad sequence index");
  if (bm->len[seq] != 0 || !bm->table[seq].empty())
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_share_prefix: sequence %d is not empty", seq);
  if (num_tokens % bm->block_size != 0 || num_tokens > bm->len[donor])
    return pa::fail(PA_ERR_INVALID_ARG,
                    "pa_bm_share_prefix: %d tokens is not a whole number of the donor's blocks",
                    num_tokens);
  const int nb = num_tokens / bm->block_size;
  bm->table[seq].assign(bm->table[donor].begin(), bm->table[donor].begin() + nb);
  for (int b : bm->table[seq]) ++bm->ref[b];
  bm->len[seq] = num_tokens;
  return PA_OK;
}

extern "C" int pa_bm_free(pa_block_manager* bm, int seq) {
  pa::clear_error();
  if (bad_seq(bm, seq)) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_free: bad sequence index");
  std::vector<int>& tab = bm->table[seq];
  for (auto it = tab.rbegin(); it != tab.rend(); ++it) drop_block(bm, *it);
  tab.clear();
  bm->len[seq] = 0;
  return PA_OK;
}

extern "C" int pa_bm_export(const pa_block_manager* bm, int32_t* block_tables,
                            int32_t* context_lens) {
  pa::clear_error();
  if (bm == nullptr || block_tables == nullptr || context_lens == nullptr)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_export: null argument");
  for (int s = 0; s < bm->max_seqs; ++s) {
    int32_t* row = block_tables + static_cast<size_t>(s) * bm->max_blocks;
    const std::vector<int>& tab = bm->table[s];
    for (int j = 0; j < bm->max_blocks; ++j) row[j] = j < static_cast<int>(tab.size()) ? tab[j] : -1;
    context_lens[s] = bm->len[s];
  }
  return PA_OK;
}
