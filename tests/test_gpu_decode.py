"""GPU parity of the CUDA path (cache write + paged decode) against the fp64
oracle, called through the C ABI on the same seeded inputs."""

import numpy as np
import pytest
import torch

from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import assert_close, int_view, oracle_decode, oracle_pools_after_write, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


# Small versions of every workload: several tiles per sequence, ragged tails,
# poisoned unused memory, the cache write first and the decode after it.
SMALL = {
    "tiny_fp32": workloads.spec("tiny_fp32"),
    "llama3_8b": workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600),
    "long_ctx": workloads.spec("long_ctx", num_seqs=2, ctx_lo=3001, ctx_hi=3001, max_context=3008, pool_blocks=0),
    "mixed_prefix": workloads.spec("mixed_prefix", num_seqs=24, ctx_median=100.0, ctx_hi=600, max_context=640,
                                   prefix_tokens=64),
    "gqa8_70b_bs16": workloads.spec("gqa8_70b", num_seqs=10, ctx_lo=1, ctx_hi=600, max_context=608),
    "gqa8_70b_bs32": workloads.spec("gqa8_70b", num_seqs=10, ctx_lo=1, ctx_hi=600, max_context=608, block_size=32),
}


def _write_then_decode(w, **decode_kw):
    g = to_device(w)
    binding.write_cache(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"])
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         **decode_kw)
    torch.cuda.synchronize()
    return g, out


@pytest.mark.parametrize("name", list(SMALL))
def test_step_parity_small(name):
    w = workloads.make_workload(SMALL[name], prewritten=False, poison=True)
    g, out = _write_then_decode(w)
    k_ref, v_ref = oracle_pools_after_write(w)
    view = int_view(w.spec.dtype)
    assert torch.equal(g["k_cache"].cpu().view(view), k_ref.view(view))
    assert torch.equal(g["v_cache"].cpu().view(view), v_ref.view(view))
    want = oracle_decode(w, k_ref, v_ref)
    assert_close(out, want, w.spec.dtype, name)


@pytest.mark.parametrize("num_ranges", [1, 2, 5, 0, 997])
@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b", "long_ctx", "mixed_prefix"])
def test_range_split_variants_agree(name, num_ranges):
    """One range (a single CTA walks every sequence, no merge) through many
    ranges (every long sequence split and merged by log-sum-exp)."""
    w = workloads.make_workload(SMALL[name], prewritten=True, poison=True)
    g = to_device(w)
    ref = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         num_ranges=1)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         num_ranges=num_ranges)
    torch.cuda.synchronize()
    want = oracle_decode(w)
    assert_close(out, want, w.spec.dtype, f"{name} R={num_ranges}")
    # Split and unsplit differ only by fp32 rounding before the output cast.
    diff = (out.double() - ref.double()).abs().max().item()
    assert diff <= (2e-6 if w.spec.dtype == "f32" else 1.6e-2), diff


EDGE_CTX = [1, 15, 16, 17, 31, 32, 33, 47, 48, 49, 0, 255, 256, 257, 2, 0]


# Block sizes cover every tensor-copy box height gcd(bs, 16): 16, 8, 4 (12), 1 (1, 3).
@pytest.mark.parametrize("block_size", [16, 32, 8, 1, 64, 3, 12, 24])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_context_lengths(block_size, dtype):
    sp = workloads.spec("llama3_8b", dtype=dtype, num_seqs=len(EDGE_CTX), max_context=272, pool_blocks=0,
                        block_size=block_size)
    w = workloads.make_workload(sp, prewritten=True, poison=True, context_lens=np.array(EDGE_CTX))
    g = to_device(w)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    want = oracle_decode(w)
    assert_close(out, want, dtype, f"bs={block_size}")
    for s, c in enumerate(EDGE_CTX):
        if c == 0:
            assert torch.all(out[s] == 0)


@pytest.mark.parametrize(
    "heads, kv_heads, head_size",
    [(8, 8, 64), (8, 8, 128), (32, 8, 128), (64, 8, 128), (16, 2, 64), (8, 1, 128), (4, 4, 128),
     (32, 16, 128), (48, 16, 64), (6, 2, 128), (7, 1, 64), (12, 12, 128), (24, 12, 64)],
)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_head_geometry(heads, kv_heads, head_size, dtype):
    sp = workloads.spec("llama3_8b", dtype=dtype, num_seqs=5, num_heads=heads, num_kv_heads=kv_heads,
                        head_size=head_size, ctx_lo=1, ctx_hi=180, max_context=192, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=True, poison=True)
    g = to_device(w)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert_close(out, oracle_decode(w), dtype, f"H={heads} Hk={kv_heads} D={head_size}")


def test_context_one_returns_v_exactly():
    """ctx = 1: each output row is the (bf16) V row itself."""
    sp = workloads.spec("gqa8_70b", num_seqs=9, max_context=16, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=True, context_lens=np.ones(9, dtype=np.int64))
    g = to_device(w)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    G = sp.num_heads // sp.num_kv_heads
    for s in range(9):
        v0 = w.v_cache[int(w.block_tables[s, 0]), 0]  # [Hk, D]
        assert torch.equal(out[s].cpu(), v0.repeat_interleave(G, 0))


def test_shared_prefix_blocks_equal_private_copies():
    """Prefix sequences reading one set of physical blocks give the same output
    as the same data stored in private blocks."""
    sp = workloads.spec("mixed_prefix", num_seqs=8, ctx_median=60.0, ctx_hi=300, max_context=320, prefix_tokens=64)
    w = workloads.make_workload(sp, prewritten=True)
    g = to_device(w)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    # Un-share: give every sequence its own copy of the prefix blocks.
    bt = w.block_tables.clone()
    pb = sp.prefix_tokens // sp.block_size
    kc, vc = [w.k_cache], [w.v_cache]
    nxt = w.num_blocks
    for s in range(0, sp.num_seqs, 2):
        ids = bt[s, :pb].long()
        kc.append(w.k_cache[ids])
        vc.append(w.v_cache[ids])
        bt[s, :pb] = torch.arange(nxt, nxt + pb, dtype=torch.int32)
        nxt += pb
    kc2, vc2 = torch.cat(kc).cuda(), torch.cat(vc).cuda()
    out2 = binding.decode(g["q"], kc2, vc2, bt.cuda(), g["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_decode_ws_matches_and_checks_size():
    w = workloads.make_workload(SMALL["llama3_8b"], prewritten=True)
    g = to_device(w)
    S, H, D = w.q.shape
    Hk = w.spec.num_kv_heads
    need = binding.pa_decode_workspace_size(S, H, Hk, D)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(g["q"])
    binding.pa_decode_ws(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], S, H, Hk,
                         D, w.spec.block_size, w.max_blocks_per_seq, w.scale, None, None, ws, need)
    ref = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # Every call leaves the merge tickets zeroed, so the scratch is reusable as is.
    tickets = (4 * S * Hk + 255) // 256 * 256  # the tickets live in the workspace's last bytes
    assert int(ws[need - tickets:].view(torch.int32).abs().sum()) == 0
    binding.pa_decode_ws(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], S, H, Hk,
                         D, w.spec.block_size, w.max_blocks_per_seq, w.scale, None, None, ws, need)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    with pytest.raises(binding.PagedAttnError) as e:
        binding.pa_decode_ws(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], S, H,
                             Hk, D, w.spec.block_size, w.max_blocks_per_seq, w.scale, None, None, ws, need - 256)
    assert e.value.code == binding.PA_ERR_WORKSPACE


def test_bad_block_id_is_reported_not_read():
    """With the bounds check on, an out-of-pool block id sets the error bit and
    the row is skipped; other sequences are unaffected."""
    w = workloads.make_workload("tiny_fp32", prewritten=True)
    g = to_device(w)
    g["block_tables"][0, 0] = w.num_blocks + 1000
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         error_flag=flag, check_block_ids=True)
    torch.cuda.synchronize()
    assert int(flag.item()) & binding.PA_DEVERR_BLOCK_ID
    want = oracle_decode(w, seqs=[1, 2, 3])
    assert_close(out[1:], want, "f32", "unaffected sequences")


def test_context_beyond_table_is_clamped_and_reported():
    w = workloads.make_workload("tiny_fp32", prewritten=True)
    g = to_device(w)
    g["context_lens"][2] = w.max_blocks_per_seq * w.spec.block_size + 7
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         error_flag=flag, check_block_ids=True)
    torch.cuda.synchronize()
    assert int(flag.item()) & binding.PA_DEVERR_CONTEXT_LEN
    assert_close(out[[0, 1, 3]], oracle_decode(w, seqs=[0, 1, 3]), "f32", "other sequences")


def test_all_sequences_empty():
    w = workloads.make_workload("tiny_fp32", prewritten=True, context_lens=np.zeros(4, dtype=np.int64))
    g = to_device(w)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         out=torch.full_like(g["q"], float("nan")))
    torch.cuda.synchronize()
    assert torch.all(out == 0)


# ---- full-size workloads, in the launch configuration the benchmark times ----

FULL = [("llama3_8b", None, [0, 7, 21, 40, 63]), ("long_ctx", None, [0, 5]),
        ("mixed_prefix", None, [0, 1, 2, 77, 150, 255]), ("gqa8_70b", 16, [0, 31, 64, 127]),
        ("gqa8_70b", 32, [3, 64, 100])]


@pytest.mark.parametrize("name, bs, sample", FULL)
def test_full_size_sampled(name, bs, sample):
    """Every full-size batch in both launch forms: the fused step the benchmark
    times (pa_decode_append, one launch) and pa_write_cache + pa_decode.  The
    two give bit-identical pools and outputs; the written rows are the new
    tokens bit for bit; sampled sequences (the longest always among them)
    match the oracle."""
    w = workloads.make_workload(name, block_size=bs, prewritten=False)
    g, out = _write_then_decode(w)
    f = to_device(w)
    out_f = binding.decode_append(f["q"], f["k_new"], f["v_new"], f["k_cache"], f["v_cache"], f["block_tables"],
                                  f["context_lens"], w.scale)
    torch.cuda.synchronize()
    view = int_view(w.spec.dtype)
    assert torch.equal(out_f.view(view), out.view(view))
    assert torch.equal(f["k_cache"].view(view), g["k_cache"].view(view))
    assert torch.equal(f["v_cache"].view(view), g["v_cache"].view(view))
    del f
    # Written rows are the new tokens, bit for bit.
    b = w.spec.block_size
    for s in sample:
        slot = int(w.slot_mapping[s])
        assert torch.equal(g["k_cache"][slot // b, slot % b].cpu().view(view), w.k_new[s].view(view))
        assert torch.equal(g["v_cache"][slot // b, slot % b].cpu().view(view), w.v_new[s].view(view))
    del g
    k_ref, v_ref = oracle_pools_after_write(w)
    # Longest sequence always in the sample.
    longest = int(torch.argmax(w.context_lens))
    sample = sorted(set(sample) | {longest})
    want = oracle_decode(w, k_ref, v_ref, seqs=sample)
    assert_close(out[sample], want, w.spec.dtype, name)
    assert_close(out_f[sample], want, w.spec.dtype, name + " (fused step)")
    assert torch.isfinite(out).all()
