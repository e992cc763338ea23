"""Reference oracle for paged decode attention and the KV-cache scatter.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may call it.  It shares no code with the CUDA path.

Everything here is a plain, slow, literal restatement of what the source pages
describe, evaluated in float64 on the exact input values (bf16 inputs are
widened exactly by the caller before they reach these functions):

* Pages cited (title, section):
  - "vLLM three-process architecture and the PagedAttention kernel"
    (devpress.csdn.net/awstech), section 3 "PagedAttention 内核原理：从概念到
    CUDA 实现": 3.1 "输入是什么" (the tensors and their shapes) and
    3.2 "内核执行流程（简化版）" steps 1-5 (look up the block table, fix the valid
    length, gather K/V through the table into a logically contiguous K_seq/V_seq,
    run standard attention with the step's query, write the output).
    Section 2 "工作流程拆解", item 4: a new token is appended to the sequence and
    gets a new physical block when the current one is full (the cache write).
  - "前言：走进 LLM 推理引擎的心脏" (vLLM book preface, yangyitao.com), section
    "从 OS 到 GPU": KV cache split into fixed-size blocks mapped on demand.
  - "vLLM LLM inference engine" course (aiflowlearn.net), section
    "KV Cache 如何被切分成页": 16 tokens per block.

Readings where the pages are silent (each is also listed in the design notes):
  - the pool is 4-D ``[num_blocks, block_size, num_kv_heads, head_size]``;
  - query head ``h`` reads KV head ``h // (num_heads // num_kv_heads)``;
  - ``context_len`` counts every valid token, the current step's included; a
    context of 0 gives an all-zero output;
  - a negative slot in ``slot_mapping`` is a padding token and is skipped;
  - the split/merge form (partial max, sum and weighted values per partition,
    combined by log-sum-exp) is the standard rescaling identity of softmax; the
    pages only say the attention "may fuse FlashAttention techniques".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "write_cache",
    "gather_sequence",
    "attention_weights",
    "attention",
    "decode",
    "decode_partials",
    "merge_partials",
    "decode_split",
    "decode_multi",
]


def write_cache(k_cache, v_cache, k_new, v_new, slot_mapping, block_size):
    """Scatter one step's new K/V rows into the paged pool (returns copies).

    Follows "vLLM three-process architecture ..." section 2 item 4 (the new
    token is appended into the sequence's current physical block) with the
    slot reading: slot ``i`` lives in block ``slot // block_size`` at offset
    ``slot % block_size``.  Works on any dtype (a byte copy), so bf16 pools can
    be passed as int16/uint16 views and compared bit for bit.

    k_cache, v_cache : [num_blocks, block_size, num_kv_heads, head_size]
    k_new, v_new     : [num_tokens, num_kv_heads, head_size]
    slot_mapping     : [num_tokens] integer; negative entries are skipped.
    """
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    for i, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        block, offset = divmod(int(slot), int(block_size))
        k_out[block, offset] = k_new[i]
        v_out[block, offset] = v_new[i]
    return k_out, v_out


def gather_sequence(cache, block_table_row, context_len, block_size):
    """Collect one sequence's K (or V) rows into a contiguous [ctx, Hk, D] array.

    Section 3.2 steps 1-3 of "vLLM three-process architecture ...": read the
    sequence's block table, derive how many logical blocks the valid length
    covers, and follow each entry to its physical block.  Token ``t`` sits in
    logical block ``t // block_size`` at offset ``t % block_size``.
    Table entries past the last needed block are never read.
    """
    ctx = int(context_len)
    num_blocks = cache.shape[0]
    flat = np.asarray(cache).reshape(num_blocks * block_size, *cache.shape[2:])
    idx = [int(block_table_row[t // block_size]) * block_size + t % block_size for t in range(ctx)]
    return flat[np.asarray(idx, dtype=np.int64)] if ctx else flat[:0]


def attention_weights(q_s, k_s, scale):
    """Softmax weights p[h, t] of one decode query over its gathered keys.

    q_s : [H, D] float64; k_s : [ctx, Hk, D] float64.  Query head h reads KV
    head h // (H // Hk).  Scores are ``scale * <q_h, k_t>``; the softmax is
    the textbook one, with the row maximum subtracted for range only.
    """
    num_heads = q_s.shape[0]
    num_kv_heads = k_s.shape[1]
    group = num_heads // num_kv_heads
    ctx = k_s.shape[0]
    p = np.zeros((num_heads, ctx), dtype=np.float64)
    if ctx == 0:
        return p
    for h in range(num_heads):
        kv = h // group
        x = scale * (k_s[:, kv, :] @ q_s[h])
        e = np.exp(x - x.max())
        p[h] = e / e.sum()
    return p


def attention(q_s, k_s, v_s, scale):
    """Standard attention of one decode query (section 3.2 step 4): sum_t p[h,t] v_t."""
    num_heads, head_size = q_s.shape
    num_kv_heads = k_s.shape[1]
    group = num_heads // num_kv_heads
    out = np.zeros((num_heads, head_size), dtype=np.float64)
    if k_s.shape[0] == 0:
        return out
    p = attention_weights(q_s, k_s, scale)
    for h in range(num_heads):
        out[h] = p[h] @ v_s[:, h // group, :]
    return out


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, block_size):
    """Paged decode attention for a batch; returns out[S, H, D] in float64.

    For each sequence: gather its K/V through its block table, then run
    attention with its query (section 3.2 steps 1-5).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    num_seqs = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(num_seqs):
        ctx = int(context_lens[s])
        k_s = gather_sequence(k_cache, block_tables[s], ctx, block_size)
        v_s = gather_sequence(v_cache, block_tables[s], ctx, block_size)
        out[s] = attention(q[s], k_s, v_s, scale)
    return out


def decode_partials(q_s, k_s, v_s, scale, partition_tokens):
    """Per-partition softmax statistics of one sequence.

    The gathered context is cut into consecutive partitions of
    ``partition_tokens`` tokens.  For partition j and head h this returns the
    partition's score maximum m[j,h], its sum of exp(score - m) l[j,h], and the
    un-normalised weighted value sum o[j,h,:] = sum_t exp(score_t - m) v_t.
    """
    num_heads, head_size = q_s.shape
    num_kv_heads = k_s.shape[1]
    group = num_heads // num_kv_heads
    ctx = k_s.shape[0]
    n_part = (ctx + partition_tokens - 1) // partition_tokens
    m = np.zeros((n_part, num_heads))
    l = np.zeros((n_part, num_heads))
    o = np.zeros((n_part, num_heads, head_size))
    for j in range(n_part):
        lo, hi = j * partition_tokens, min(ctx, (j + 1) * partition_tokens)
        for h in range(num_heads):
            kv = h // group
            x = scale * (k_s[lo:hi, kv, :] @ q_s[h])
            m[j, h] = x.max()
            e = np.exp(x - m[j, h])
            l[j, h] = e.sum()
            o[j, h] = e @ v_s[lo:hi, kv, :]
    return m, l, o


def merge_partials(m, l, o):
    """Log-sum-exp merge: out = sum_j exp(m_j - M) o_j / sum_j exp(m_j - M) l_j."""
    big_m = m.max(axis=0)
    w = np.exp(m - big_m[None, :])
    num = (w[:, :, None] * o).sum(axis=0)
    den = (w * l).sum(axis=0)
    return num / den[:, None]


def decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, block_size, partition_tokens):
    """Same result as :func:`decode`, computed partition by partition and merged."""
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(q.shape[0]):
        ctx = int(context_lens[s])
        if ctx == 0:
            continue
        k_s = gather_sequence(k_cache, block_tables[s], ctx, block_size)
        v_s = gather_sequence(v_cache, block_tables[s], ctx, block_size)
        m, l, o = decode_partials(q[s], k_s, v_s, scale, partition_tokens)
        out[s] = merge_partials(m, l, o)
    return out



def decode_multi(q, k_cache, v_cache, block_tables, context_lens, scale, block_size):
    """Several new query tokens per sequence over the paged cache, causal.

    q : [S, Q, H, D].  The Q newest tokens of sequence s (already in the cache,
    context_lens[s] counting them) sit at positions c - Q + i, i < Q; query i
    attends to the gathered keys 0..c - Q + i (a causal mask over the
    sequence).  A query whose position is negative (c < Q) has no keys and
    gives zeros.  Returns out[S, Q, H, D] in float64.

    This extends the decode step of "vLLM three-process architecture and the
    PagedAttention kernel" section 3.2 (gather through the block table, then
    standard attention) to the several-token steps the pages name: chunked
    prefill and speculative-decoding verification (vLLM book preface, reader
    questions; the is96 essay's feature list).
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    num_seqs, num_q = q.shape[:2]
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(num_seqs):
        ctx = int(context_lens[s])
        k_s = gather_sequence(k_cache, block_tables[s], ctx, block_size)
        v_s = gather_sequence(v_cache, block_tables[s], ctx, block_size)
        for i in range(num_q):
            pos = ctx - num_q + i
            if pos < 0:
                continue
            out[s, i] = attention(q[s, i], k_s[: pos + 1], v_s[: pos + 1], scale)
    return out
