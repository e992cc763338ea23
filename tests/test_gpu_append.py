"""GPU parity of pa_decode_append (the cache write fused into the decode): its
output and pools equal pa_write_cache followed by pa_decode bit for bit, and
the output matches the fp64 oracle on the written pools."""

import numpy as np
import pytest
import torch

from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import assert_close, oracle_decode, oracle_pools_after_write, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


CASES = {
    "llama3_8b": workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600),
    "gqa8_70b": workloads.spec("gqa8_70b", num_seqs=10, ctx_lo=1, ctx_hi=600, max_context=608),
    "two_head_groups": workloads.spec("llama3_8b", num_seqs=6, num_heads=32, num_kv_heads=16, ctx_lo=1,
                                      ctx_hi=300, max_context=320, pool_blocks=0),
    "d64": workloads.spec("gqa8_70b", num_seqs=6, ctx_lo=1, ctx_hi=300, max_context=304, head_size=64),
    "bs1": workloads.spec("llama3_8b", num_seqs=5, ctx_lo=1, ctx_hi=90, max_context=96, pool_blocks=0,
                          block_size=1),
    "bs24": workloads.spec("llama3_8b", num_seqs=8, ctx_lo=1, ctx_hi=400, max_context=408, pool_blocks=0,
                           block_size=24),
}


def _both(w, **kw):
    a = to_device(w)
    binding.write_cache(a["k_new"], a["v_new"], a["slot_mapping"], a["k_cache"], a["v_cache"])
    out_a = binding.decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"], w.scale, **kw)
    b = to_device(w)
    out_b = binding.decode_append(b["q"], b["k_new"], b["v_new"], b["k_cache"], b["v_cache"], b["block_tables"],
                                  b["context_lens"], w.scale, **kw)
    torch.cuda.synchronize()
    return a, out_a, b, out_b


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("num_ranges", [0, 1, 5, 997])
def test_append_equals_write_then_decode(name, num_ranges):
    w = workloads.make_workload(CASES[name], prewritten=False, poison=True)
    a, out_a, b, out_b = _both(w, num_ranges=num_ranges, check_block_ids=True)
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))
    assert torch.equal(b["k_cache"].view(torch.int16), a["k_cache"].view(torch.int16))
    assert torch.equal(b["v_cache"].view(torch.int16), a["v_cache"].view(torch.int16))
    k_ref, v_ref = oracle_pools_after_write(w)
    assert torch.equal(b["k_cache"].cpu().view(torch.int16), k_ref.view(torch.int16))
    assert_close(out_b, oracle_decode(w, k_ref, v_ref), "bf16", f"append {name} R={num_ranges}")


EDGE_CTX = [1, 15, 16, 17, 31, 32, 33, 0, 255, 256, 257, 2, 0]


def test_append_edge_contexts():
    sp = workloads.spec("llama3_8b", num_seqs=len(EDGE_CTX), max_context=272, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=False, poison=True, context_lens=np.array(EDGE_CTX))
    a, out_a, b, out_b = _both(w)
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))
    assert torch.equal(b["k_cache"].view(torch.int16), a["k_cache"].view(torch.int16))
    assert torch.equal(b["v_cache"].view(torch.int16), a["v_cache"].view(torch.int16))
    for s, c in enumerate(EDGE_CTX):
        if c == 0:
            assert torch.all(out_b[s] == 0)


def test_append_steps_match_separate_write():
    """Several steps in a row: each step's newest token lands where the next
    step reads it, exactly as with the separate cache write."""
    sp = CASES["llama3_8b"]
    w = workloads.make_workload(sp, prewritten=False, poison=True)
    a, b = to_device(w), to_device(w)
    gen = torch.Generator().manual_seed(9)
    lens = w.context_lens.clone()
    bs = sp.block_size
    bt = w.block_tables
    for step in range(4):
        kn = torch.randn(w.k_new.shape, generator=gen).to(torch.bfloat16).cuda()
        vn = torch.randn(w.v_new.shape, generator=gen).to(torch.bfloat16).cuda()
        if step > 0:
            # A sequence grows by one token when that token's block is already
            # in its table; otherwise its newest token is rewritten in place.
            lens = torch.tensor([c + 1 if c // bs < bt.shape[1] and int(bt[s, c // bs]) >= 0 else c
                                 for s, c in enumerate(lens.tolist())], dtype=lens.dtype)
        slots = torch.tensor([int(bt[s, (c - 1) // bs]) * bs + (c - 1) % bs if c > 0 else -1
                              for s, c in enumerate(lens.tolist())], dtype=torch.int64)
        ld = lens.cuda()
        binding.write_cache(kn, vn, slots.cuda(), a["k_cache"], a["v_cache"])
        out_a = binding.decode(a["q"], a["k_cache"], a["v_cache"], a["block_tables"], ld, w.scale)
        out_b = binding.decode_append(b["q"], kn, vn, b["k_cache"], b["v_cache"], b["block_tables"], ld, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16)), step
        assert torch.equal(b["k_cache"].view(torch.int16), a["k_cache"].view(torch.int16)), step
        assert torch.equal(b["v_cache"].view(torch.int16), a["v_cache"].view(torch.int16)), step


def test_append_rejects_fp32():
    w = workloads.make_workload("tiny_fp32", prewritten=False)
    g = to_device(w)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.decode_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], w.scale)
    assert e.value.code == binding.PA_ERR_UNSUPPORTED
