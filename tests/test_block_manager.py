"""Host block manager (pa_bm_*): free pool, on-demand blocks, reference
counts with copy-on-write, prefix sharing, reuse of freed blocks.  Host
memory only, so these run without a GPU."""

import random

import pytest

from paged_kv_cache_292_gb300 import binding
from paged_kv_cache_292_gb300 import build as pa_build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    binding.load()


def test_on_demand_blocks_and_slots():
    bm = binding.BlockManager(10, 4, 3, 5)
    slots, copies = bm.append(0, 6)
    assert slots.tolist() == [0, 1, 2, 3, 4, 5] and copies == []  # blocks 0 and 1, in pool order
    assert bm.num_free_blocks() == 8 and bm.context_len(0) == 6
    slots, _ = bm.append(0, 3)  # 2 more fill block 1, the third opens block 2
    assert slots.tolist() == [6, 7, 8]
    tables, lens = bm.export()
    assert tables[0].tolist() == [0, 1, 2, -1, -1] and lens.tolist() == [9, 0, 0]


def test_fork_then_copy_on_write_of_a_shared_partial_block():
    bm = binding.BlockManager(10, 4, 3, 5)
    bm.append(0, 6)  # blocks 0, 1 (block 1 half full)
    bm.fork(0, 1)
    assert bm.ref_count(0) == 2 and bm.ref_count(1) == 2
    slots, copies = bm.append(1, 1)  # child writes into the shared half-full block
    assert copies == [(1, 2)]  # private copy of block 1 in block 2
    assert slots.tolist() == [2 * 4 + 2]
    tables, lens = bm.export()
    assert tables[0].tolist()[:2] == [0, 1] and tables[1].tolist()[:2] == [0, 2]
    assert bm.ref_count(1) == 1 and bm.ref_count(2) == 1 and bm.ref_count(0) == 2
    # The parent's block is now private again: no copy on its next append.
    _, copies = bm.append(0, 1)
    assert copies == []


def test_no_copy_when_the_shared_last_block_is_full():
    bm = binding.BlockManager(10, 4, 3, 5)
    bm.append(0, 8)  # two full blocks
    bm.fork(0, 1)
    slots, copies = bm.append(1, 1)
    assert copies == [] and slots.tolist() == [2 * 4]


def test_prefix_sharing_whole_blocks_only():
    bm = binding.BlockManager(12, 4, 3, 6)
    bm.append(0, 10)
    bm.share_prefix(1, 0, 8)
    tables, lens = bm.export()
    assert tables[1].tolist()[:2] == tables[0].tolist()[:2] and lens[1] == 8
    assert bm.ref_count(int(tables[0][0])) == 2
    slots, copies = bm.append(1, 1)  # prefix ends on a block boundary: a fresh block
    assert copies == [] and int(slots[0]) // 4 not in tables[0].tolist()
    with pytest.raises(binding.PagedAttnError):
        bm.share_prefix(2, 0, 6)  # not a whole number of blocks


def test_free_returns_blocks_first_in_line():
    bm = binding.BlockManager(6, 4, 3, 4)
    bm.append(0, 8)  # blocks 0, 1
    bm.append(1, 4)  # block 2
    bm.free(0)
    assert bm.num_free_blocks() == 5
    slots, _ = bm.append(2, 8)
    assert sorted({int(s) // 4 for s in slots}) == [0, 1]  # the freed blocks are reused at once


def test_errors_leave_state_unchanged():
    bm = binding.BlockManager(3, 4, 2, 8)
    bm.append(0, 8)
    with pytest.raises(binding.PagedAttnError) as e:
        bm.append(1, 9)  # needs 3 blocks, 1 free
    assert e.value.code == binding.PA_ERR_NO_BLOCKS
    assert bm.num_free_blocks() == 1 and bm.context_len(1) == 0
    bm2 = binding.BlockManager(20, 4, 2, 2)
    with pytest.raises(binding.PagedAttnError) as e:
        bm2.append(0, 9)  # 3 blocks > max_blocks_per_seq
    assert e.value.code == binding.PA_ERR_INVALID_ARG
    with pytest.raises(binding.PagedAttnError):
        bm.fork(0, 0)
    with pytest.raises(binding.PagedAttnError):
        bm.fork(5, 1)


class _Model:
    """Independent pure-Python statement of the same allocation rules."""

    def __init__(self, nb, bs, seqs, mb):
        self.bs, self.mb = bs, mb
        self.free = list(range(nb))
        self.ref = [0] * nb
        self.tab = [[] for _ in range(seqs)]
        self.len = [0] * seqs

    def append(self, s, n):
        cur, want = self.len[s], self.len[s] + n
        need = -(-want // self.bs)
        if need > self.mb:
            return "invalid", None
        cow = n > 0 and cur % self.bs and self.ref[self.tab[s][-1]] > 1
        fresh = need - len(self.tab[s]) + (1 if cow else 0)
        if fresh > len(self.free):
            return "noblocks", None
        copies = []
        if cow:
            old, new = self.tab[s][-1], self.free.pop(0)
            self.ref[new] = 1
            self.ref[old] -= 1
            if self.ref[old] == 0:
                self.free.insert(0, old)
            self.tab[s][-1] = new
            copies = [(old, new)]
        while len(self.tab[s]) < need:
            b = self.free.pop(0)
            self.ref[b] = 1
            self.tab[s].append(b)
        self.len[s] = want
        return [self.tab[s][t // self.bs] * self.bs + t % self.bs for t in range(cur, want)], copies

    def fork(self, p, c):
        self.tab[c] = list(self.tab[p])
        for b in self.tab[c]:
            self.ref[b] += 1
        self.len[c] = self.len[p]

    def free_seq(self, s):
        for b in reversed(self.tab[s]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.insert(0, b)
        self.tab[s], self.len[s] = [], 0


@pytest.mark.parametrize("seed", range(4))
def test_random_operations_match_a_reference_model(seed):
    rng = random.Random(seed)
    nb, bs, seqs, mb = 40, rng.choice([1, 3, 4, 16]), 6, 12
    bm = binding.BlockManager(nb, bs, seqs, mb)
    model = _Model(nb, bs, seqs, mb)
    for _ in range(300):
        op = rng.random()
        s = rng.randrange(seqs)
        if op < 0.6:
            n = rng.randrange(0, 2 * bs + 2)
            want, copies = model.append(s, n)
            if isinstance(want, str):
                with pytest.raises(binding.PagedAttnError):
                    bm.append(s, n)
            else:
                slots, got_copies = bm.append(s, n)
                assert slots.tolist() == want and got_copies == copies
        elif op < 0.75:
            c = rng.randrange(seqs)
            if c != s and model.len[c] == 0 and not model.tab[c]:
                bm.fork(s, c)
                model.fork(s, c)
        else:
            bm.free(s)
            model.free_seq(s)
        assert bm.num_free_blocks() == len(model.free)
        tables, lens = bm.export()
        for q in range(seqs):
            assert tables[q].tolist()[: len(model.tab[q])] == model.tab[q]
            assert int(lens[q]) == model.len[q]
        assert all(bm.ref_count(b) == model.ref[b] for b in range(nb))


def test_append_batch_equals_single_appends():
    a = binding.BlockManager(50, 4, 4, 10)
    b = binding.BlockManager(50, 4, 4, 10)
    for m in (a, b):
        m.append(0, 6)
        m.fork(0, 1)
    slots_a, copies_a = a.append_batch([0, 1, 2, 3], [1, 2, 5, 0])
    want, copies_b = [], []
    for s, n in zip([0, 1, 2, 3], [1, 2, 5, 0]):
        sl, cp = b.append(s, n)
        want += sl.tolist()
        copies_b += cp
    assert slots_a.tolist() == want and copies_a == copies_b
