"""GPU parity of pa_decode_mq_append (several query tokens per sequence with
their cache write fused into the decode): output and pools equal
pa_write_cache of the Q new rows followed by pa_decode_mq bit for bit, the
pools equal the generator's (the new rows are the values it placed there
before they were poisoned), and the output matches the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


def _case(sp, Q, context_lens=None):
    """Pools holding every token, the Q newest rows of each sequence lifted out
    into k_new / v_new ([S*Q, Hk, D]) and replaced by NaN in the pools."""
    w = workloads.make_workload(sp, prewritten=True, poison=True, context_lens=context_lens)
    S, H, D = w.q.shape
    bs = sp.block_size
    rng = np.random.default_rng([sp.seed, 78, Q])
    q = torch.from_numpy(rng.standard_normal((S, Q, H, D), dtype=np.float32)).to(w.q.dtype)
    Hk = w.k_cache.shape[2]
    k_new = torch.from_numpy(rng.standard_normal((S * Q, Hk, D), dtype=np.float32)).to(w.k_cache.dtype)
    v_new = torch.from_numpy(rng.standard_normal((S * Q, Hk, D), dtype=np.float32)).to(w.k_cache.dtype)
    slots = np.full(S * Q, -1, dtype=np.int64)
    k0, v0 = w.k_cache.clone(), w.v_cache.clone()
    for s, c in enumerate(w.context_lens.tolist()):
        for i in range(Q):
            pos = c - Q + i
            if pos < 0:
                continue  # the query's token precedes the sequence: nothing to write
            blk, off = int(w.block_tables[s, pos // bs]), pos % bs
            slots[s * Q + i] = blk * bs + off
            k_new[s * Q + i] = w.k_cache[blk, off]
            v_new[s * Q + i] = w.v_cache[blk, off]
            k0[blk, off] = float("nan")
            v0[blk, off] = float("nan")
    return w, q, k_new, v_new, torch.from_numpy(slots), k0, v0


def _oracle(w, q):
    return oracle.decode_multi(q.double().numpy(), w.k_cache.double().numpy(), w.v_cache.double().numpy(),
                               w.block_tables.numpy(), w.context_lens.numpy(), w.scale, w.spec.block_size)


def _check(sp, Q, num_ranges=0, context_lens=None, what=""):
    w, q, k_new, v_new, slots, k0, v0 = _case(sp, Q, context_lens)
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    qd, kn, vn = q.cuda(), k_new.cuda(), v_new.cuda()
    ka, va = k0.cuda(), v0.cuda()
    binding.write_cache(kn, vn, slots.cuda(), ka, va)
    out_a = binding.decode_multi(qd, ka, va, bt, cl, w.scale, num_ranges=num_ranges)
    kb, vb = k0.cuda(), v0.cuda()
    out_b = binding.decode_multi_append(qd, kn, vn, kb, vb, bt, cl, w.scale, num_ranges=num_ranges,
                                        check_block_ids=True)
    torch.cuda.synchronize()
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16)), what
    assert torch.equal(kb.view(torch.int16), ka.view(torch.int16)), what
    assert torch.equal(vb.view(torch.int16), va.view(torch.int16)), what
    assert torch.equal(kb.cpu().view(torch.int16), w.k_cache.view(torch.int16)), what
    assert torch.equal(vb.cpu().view(torch.int16), w.v_cache.view(torch.int16)), what
    assert_close(out_b, _oracle(w, q), "bf16", what)


SMALL_LLAMA = dict(num_seqs=10, ctx_lo=1, ctx_hi=500, max_context=512, pool_blocks=0)


@pytest.mark.parametrize("Q", [1, 2, 4])
@pytest.mark.parametrize("num_ranges", [0, 1, 5, 997])
def test_mq_append_llama_shaped(Q, num_ranges):
    _check(workloads.spec("llama3_8b", **SMALL_LLAMA), Q, num_ranges, what=f"Q={Q} R={num_ranges}")


@pytest.mark.parametrize("Q", [2, 3])
@pytest.mark.parametrize("block_size", [8, 1, 24])
def test_mq_append_block_sizes(Q, block_size):
    _check(workloads.spec("llama3_8b", **dict(SMALL_LLAMA, block_size=block_size)), Q, what=f"Q={Q} bs={block_size}")


# More than 8 (query, head) columns per KV head (two to four warps per KV
# head): the rows are written by their own kernel ahead of the decode.
@pytest.mark.parametrize("heads, kv_heads, Q", [(8, 1, 2), (10, 2, 3), (32, 8, 3), (64, 8, 2), (64, 8, 3),
                                                 (64, 8, 4), (32, 8, 5)])
@pytest.mark.parametrize("num_ranges", [0, 1, 5])
def test_mq_append_split_columns(heads, kv_heads, Q, num_ranges):
    sp = workloads.spec("llama3_8b", num_heads=heads, num_kv_heads=kv_heads, num_seqs=7, ctx_lo=1, ctx_hi=300,
                        max_context=304, pool_blocks=0)
    _check(sp, Q, num_ranges, what=f"H={heads} Hk={kv_heads} Q={Q} R={num_ranges}")


def test_mq_append_head_size_64():
    sp = workloads.spec("gqa8_70b", num_seqs=6, ctx_lo=1, ctx_hi=300, max_context=304, head_size=64)
    _check(sp, 2, what="D=64")


# New tokens that straddle tile and block boundaries, and contexts shorter than Q.
EDGE_CTX = [1, 2, 3, 4, 15, 16, 17, 18, 31, 32, 33, 0, 255, 256, 257, 258]


@pytest.mark.parametrize("Q", [2, 4])
def test_mq_append_edge_contexts(Q):
    sp = workloads.spec("llama3_8b", num_seqs=len(EDGE_CTX), max_context=272, pool_blocks=0)
    _check(sp, Q, context_lens=np.array(EDGE_CTX), what=f"edges Q={Q}")
