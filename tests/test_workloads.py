"""Structure of the seeded decode batches (CPU only)."""

import numpy as np
import pytest
import torch

from paged_kv_cache_292_gb300 import workloads


def _small(name):
    if name == "tiny_fp32":
        return workloads.spec(name)
    if name == "mixed_prefix":
        return workloads.spec(name, num_seqs=10, ctx_median=40.0, ctx_hi=256, max_context=256, prefix_tokens=64)
    return workloads.spec(name, num_seqs=5, ctx_lo=1, ctx_hi=100, max_context=112, pool_blocks=0)


@pytest.mark.parametrize("name", list(workloads.SPECS))
def test_shapes_and_determinism(name):
    sp = _small(name)
    a = workloads.make_workload(sp)
    b = workloads.make_workload(sp)
    S, H, Hk, D, bs = sp.num_seqs, sp.num_heads, sp.num_kv_heads, sp.head_size, sp.block_size
    assert a.q.shape == (S, H, D)
    assert a.k_cache.shape == (a.num_blocks, bs, Hk, D) == a.v_cache.shape
    assert a.block_tables.shape == (S, a.max_blocks_per_seq) and a.block_tables.dtype == torch.int32
    assert a.context_lens.dtype == torch.int32 and a.slot_mapping.dtype == torch.int64
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache), (a.block_tables, b.block_tables)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("name", list(workloads.SPECS))
def test_tables_cover_context_and_slots_point_at_last_token(name):
    w = workloads.make_workload(_small(name))
    bs = w.spec.block_size
    bt = w.block_tables.numpy()
    used = []
    for s, c in enumerate(w.context_lens.tolist()):
        n = -(-c // bs)
        assert np.all(bt[s, :n] >= 0) and np.all(bt[s, :n] < w.num_blocks)
        assert np.all(bt[s, n:] == -1)
        used.extend(bt[s, :n].tolist())
        last = c - 1
        assert w.slot_mapping[s] == bt[s, last // bs] * bs + last % bs
    counts = np.bincount(used, minlength=w.num_blocks)
    # Only the shared prefix blocks may appear in more than one table.
    assert int((counts > 1).sum()) == w.shared_blocks


def test_prefix_sharing_layout():
    sp = _small("mixed_prefix")
    w = workloads.make_workload(sp)
    bt = w.block_tables.numpy()
    pb = sp.prefix_tokens // sp.block_size
    even = bt[0::2, :pb]
    assert (even == even[0]).all() and w.shared_blocks == pb
    # Odd sequences own private blocks only.
    assert not set(bt[1::2][bt[1::2] >= 0].tolist()) & set(even[0].tolist())
    # The newest token of a sharing sequence lands beyond the prefix.
    assert all(int(w.slot_mapping[s]) // sp.block_size not in set(even[0].tolist()) for s in range(0, sp.num_seqs, 2))


def test_named_specs_match_stated_sizes():
    s = workloads.SPECS
    assert (s["llama3_8b"].num_seqs, s["llama3_8b"].num_heads, s["llama3_8b"].num_kv_heads) == (64, 32, 8)
    assert s["llama3_8b"].pool_blocks == 32768 and s["llama3_8b"].max_context // 16 == 256
    assert s["long_ctx"].ctx_lo == s["long_ctx"].ctx_hi == 32768 and s["long_ctx"].num_seqs == 8
    assert s["mixed_prefix"].num_seqs == 256 and s["mixed_prefix"].prefix_tokens == 1024
    assert (s["gqa8_70b"].num_heads, s["gqa8_70b"].num_kv_heads, s["gqa8_70b"].num_seqs) == (64, 8, 128)
    assert s["tiny_fp32"].pool_blocks == 64 and s["tiny_fp32"].dtype == "f32"


def test_poison_fills_unused_slots_with_nan():
    w = workloads.make_workload("tiny_fp32", poison=True)
    bs = w.spec.block_size
    valid = torch.zeros(w.num_blocks, bs, dtype=torch.bool)
    for s, c in enumerate(w.context_lens.tolist()):
        for t in range(c):
            valid[w.block_tables[s, t // bs], t % bs] = True
    assert torch.isnan(w.k_cache[~valid]).all() and torch.isfinite(w.k_cache[valid]).all()


def test_unwritten_slot_is_left_for_the_cache_write():
    w = workloads.make_workload("tiny_fp32", prewritten=False, poison=True)
    bs = w.spec.block_size
    for s in range(w.spec.num_seqs):
        slot = int(w.slot_mapping[s])
        assert torch.isnan(w.k_cache[slot // bs, slot % bs]).all()
        assert torch.isfinite(w.k_new[s]).all()


@pytest.mark.parametrize("Q", [1, 2, 5])
def test_multi_query_step_layout(Q):
    """Q new tokens per sequence at positions ctx - Q .. ctx - 1: rows s * Q + i,
    each row's slot is that position's place in the sequence's blocks, -1
    before the sequence's start; the same draws every time."""
    ctx = np.array([1, 3, 16, 17, 40, 0])
    sp = workloads.spec("llama3_8b", num_seqs=len(ctx), max_context=48, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=False, context_lens=ctx)
    q, kn, vn, slots = workloads.multi_query_step(w, Q)
    S, H, D = w.q.shape
    assert q.shape == (S, Q, H, D) and q.dtype == w.q.dtype
    assert kn.shape == vn.shape == (S * Q, sp.num_kv_heads, D) and kn.dtype == w.k_cache.dtype
    assert slots.shape == (S * Q,) and slots.dtype == torch.int64
    bs = sp.block_size
    bt = w.block_tables.numpy()
    for s, c in enumerate(ctx):
        for i in range(Q):
            pos = int(c) - Q + i
            want = -1 if pos < 0 else int(bt[s, pos // bs]) * bs + pos % bs
            assert int(slots[s * Q + i]) == want
    again = workloads.multi_query_step(w, Q)
    assert all(torch.equal(a, b) for a, b in zip((q, kn, vn, slots), again))
    if Q == 1:
        # One query: the newest token's slot is the workload's own slot.
        assert torch.equal(slots[ctx > 0], w.slot_mapping[ctx > 0])
