"""GPU parity of the multi-query causal path (pa_decode_mq) against the fp64
oracle (decode_multi) on the same seeded inputs."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


def _case(name, Q, seed=0, **kw):
    sp = workloads.spec(name, **kw)
    w = workloads.make_workload(sp, prewritten=True, poison=True)
    S, H, D = w.q.shape
    q = torch.from_numpy(np.random.default_rng([sp.seed, 77, seed]).standard_normal((S, Q, H, D),
                                                                                   dtype=np.float32))
    q = q.to(w.q.dtype)
    return w, q


def _oracle(w, q):
    return oracle.decode_multi(q.double().numpy(), w.k_cache.double().numpy(), w.v_cache.double().numpy(),
                               w.block_tables.numpy(), w.context_lens.numpy(), w.scale, w.spec.block_size)


SMALL_LLAMA = dict(num_seqs=10, ctx_lo=1, ctx_hi=500, max_context=512, pool_blocks=400)


@pytest.mark.parametrize("Q", [1, 2, 3, 4])
@pytest.mark.parametrize("num_ranges", [0, 1, 5, 997])
def test_multi_query_llama_shaped(Q, num_ranges):
    w, q = _case("llama3_8b", Q, **SMALL_LLAMA)
    g = to_device(w)
    out = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                               num_ranges=num_ranges)
    torch.cuda.synchronize()
    assert_close(out, _oracle(w, q), "bf16", f"Q={Q} R={num_ranges}")


@pytest.mark.parametrize("Q", [1, 2, 3, 4])
@pytest.mark.parametrize("D", [64, 128])
def test_multi_query_gqa8(Q, D):
    w, q = _case("gqa8_70b", Q, num_seqs=6, ctx_lo=1, ctx_hi=300, max_context=304, head_size=D)
    g = to_device(w)
    out = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert_close(out, _oracle(w, q), "bf16", f"G=8 Q={Q} D={D}")


@pytest.mark.parametrize("Q", [2, 4])
@pytest.mark.parametrize("block_size", [8, 1, 24])
def test_multi_query_block_sizes(Q, block_size):
    w, q = _case("llama3_8b", Q, **dict(SMALL_LLAMA, block_size=block_size, pool_blocks=0))
    g = to_device(w)
    out = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert_close(out, _oracle(w, q), "bf16", f"Q={Q} bs={block_size}")


# More than 8 (query, head) columns per KV head: two to four warps per KV head
# (8 columns each), the last with padding columns when G * Q is not a multiple
# of 8: 16, 12, 15, 12, 20 (three warps), 24, 32 (four warps), 28, 32 columns.
@pytest.mark.parametrize("heads, kv_heads, Q", [(8, 1, 2), (12, 2, 2), (10, 2, 3), (32, 8, 3), (32, 8, 5),
                                                 (64, 8, 3), (64, 8, 4), (14, 2, 4), (16, 2, 4)])
@pytest.mark.parametrize("num_ranges", [0, 1, 5])
def test_multi_query_split_columns(heads, kv_heads, Q, num_ranges):
    w, q = _case("llama3_8b", Q, seed=heads, num_heads=heads, num_kv_heads=kv_heads, num_seqs=7, ctx_lo=1,
                 ctx_hi=400, max_context=400, pool_blocks=0)
    g = to_device(w)
    out = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                               num_ranges=num_ranges)
    torch.cuda.synchronize()
    assert_close(out, _oracle(w, q), "bf16", f"H={heads} Hk={kv_heads} Q={Q} R={num_ranges}")


def test_short_contexts_give_zero_rows_for_queries_before_the_start():
    ctx = np.array([1, 2, 3, 4, 5, 17])
    sp = workloads.spec("llama3_8b", num_seqs=len(ctx), max_context=32, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=True, poison=True, context_lens=ctx)
    q = torch.randn(len(ctx), 4, 32, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    g = to_device(w)
    out = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    want = _oracle(w, q)
    assert_close(out, want, "bf16", "short contexts")
    assert torch.all(out[0, :3] == 0) and torch.all(out[2, :1] == 0)


@pytest.mark.parametrize("Q", [2, 4])
def test_empty_sequences_zero_all_their_query_rows(Q):
    """A sequence with context 0 gets Q zero rows, and no other sequence's rows
    are touched (the output starts as NaN)."""
    ctx = np.array([5, 0, 40, 0, 17, 3, 0, 33])
    sp = workloads.spec("llama3_8b", num_seqs=len(ctx), max_context=48, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=True, poison=True, context_lens=ctx)
    q = torch.randn(len(ctx), Q, 32, 128, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    g = to_device(w)
    out = torch.full((len(ctx), Q, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         out=out)
    torch.cuda.synchronize()
    assert_close(out, _oracle(w, q), "bf16", f"empty sequences Q={Q}")
    for s in np.flatnonzero(ctx == 0):
        assert torch.all(out[s] == 0)


def test_one_query_equals_pa_decode():
    w, q = _case("llama3_8b", 1, **SMALL_LLAMA)
    g = to_device(w)
    a = binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    b = binding.decode(q[:, 0].contiguous().cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"],
                       w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


def test_rejects_unsupported_shapes():
    w, q = _case("llama3_8b", 9, **SMALL_LLAMA)  # G=4 x 9 queries = 36 > 32 columns
    g = to_device(w)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.decode_multi(q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    assert e.value.code == binding.PA_ERR_UNSUPPORTED
