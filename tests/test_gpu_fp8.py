"""GPU parity of the FP8 (E4M3) KV pool: the quantising cache write is
bit-exact against the oracle's encoder, and decode over FP8 pools matches the
fp64 oracle on the dequantised pools."""

import numpy as np
import pytest
import torch

from oracle import fp8 as ofp8
from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import assert_close

pytestmark = pytest.mark.gpu

NAN_CODE = 0x7F  # E4M3 NaN: poison for slots no token owns


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


def _codes_of_pool(w, pool, scale):
    """Oracle-quantised codes for every valid token; NaN codes elsewhere."""
    bs = w.spec.block_size
    codes = np.full(pool.shape, NAN_CODE, dtype=np.uint8)
    bt, ctx = w.block_tables.numpy(), w.context_lens.numpy()
    flat_c = codes.reshape(-1, *pool.shape[2:])
    flat_p = pool.float().numpy().reshape(-1, *pool.shape[2:])
    for s, c in enumerate(ctx.tolist()):
        idx = [int(bt[s, t // bs]) * bs + t % bs for t in range(c)]
        flat_c[idx] = ofp8.quantize(flat_p[idx], scale)
    return codes


@pytest.mark.parametrize("src", ["bf16", "f32"])
@pytest.mark.parametrize("k_scale, v_scale", [(1.0, 1.0), (0.37, 2.5), (1e-3, 1e-3)])
def test_fp8_write_cache_bit_exact(src, k_scale, v_scale):
    g = torch.Generator().manual_seed(4)
    nb, bs, hk, d, t = 20, 16, 8, 128, 40
    tdt = torch.bfloat16 if src == "bf16" else torch.float32
    kn = (torch.randn(t, hk, d, generator=g) * 3).to(tdt)
    vn = (torch.randn(t, hk, d, generator=g) * 3).to(tdt)
    slots = torch.randperm(nb * bs, generator=g)[:t].to(torch.int64)
    slots[5] = -1
    kc = torch.full((nb, bs, hk, d), NAN_CODE, dtype=torch.uint8)
    vc = kc.clone()
    k_ref, v_ref = ofp8.write_cache_fp8(kc.numpy(), vc.numpy(), kn.float().numpy(), vn.float().numpy(),
                                        slots.numpy(), bs, k_scale, v_scale)
    dk, dv = kc.cuda(), vc.cuda()
    binding.write_cache_fp8(kn.cuda(), vn.cuda(), slots.cuda(), dk, dv, k_scale, v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy(), k_ref)
    assert np.array_equal(dv.cpu().numpy(), v_ref)


SMALL = {
    "llama3_8b": workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600),
    "long_split": workloads.spec("long_ctx", num_seqs=2, ctx_lo=3001, ctx_hi=3001, max_context=3008, pool_blocks=0),
    "gqa8_d64": workloads.spec("gqa8_70b", num_seqs=6, ctx_lo=1, ctx_hi=300, max_context=304, head_size=64),
    "gqa8_bs32": workloads.spec("gqa8_70b", num_seqs=6, ctx_lo=1, ctx_hi=300, max_context=320, block_size=32),
    "llama_bs8": workloads.spec("llama3_8b", num_seqs=8, ctx_lo=1, ctx_hi=400, max_context=400, pool_blocks=0,
                                block_size=8),
    "llama_bs1": workloads.spec("llama3_8b", num_seqs=4, ctx_lo=1, ctx_hi=100, max_context=100, pool_blocks=0,
                                block_size=1),
    "llama_bs24": workloads.spec("llama3_8b", num_seqs=8, ctx_lo=1, ctx_hi=400, max_context=408, pool_blocks=0,
                                 block_size=24),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("num_ranges", [0, 1, 5])
def test_fp8_decode_matches_oracle(name, num_ranges):
    w = workloads.make_workload(SMALL[name], prewritten=True)
    k_scale, v_scale = 0.5, 0.25
    kcode = _codes_of_pool(w, w.k_cache, k_scale)
    vcode = _codes_of_pool(w, w.v_cache, v_scale)
    out = binding.decode_fp8(w.q.cuda(), torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda(),
                             w.block_tables.cuda(), w.context_lens.cuda(), w.scale, k_scale, v_scale,
                             num_ranges=num_ranges)
    torch.cuda.synchronize()
    want = ofp8.decode_fp8(w.q.double().numpy(), kcode, vcode, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.scale, w.spec.block_size, k_scale, v_scale)
    assert_close(out, want, "bf16", f"fp8 {name} R={num_ranges}")


def test_fp8_write_then_decode_step():
    """The whole FP8 step: quantising write of the new tokens, then decode."""
    sp = SMALL["llama3_8b"]
    w = workloads.make_workload(sp, prewritten=False)
    k_scale, v_scale = 1.0, 1.0
    kcode = _codes_of_pool(w, w.k_cache, k_scale)  # positions 0..c-2 (the newest token is not in the pool yet)
    vcode = _codes_of_pool(w, w.v_cache, v_scale)
    bs = sp.block_size
    for s, c in enumerate(w.context_lens.tolist()):  # the newest slot holds poison until written
        slot = int(w.slot_mapping[s])
        kcode[slot // bs, slot % bs] = NAN_CODE
        vcode[slot // bs, slot % bs] = NAN_CODE
    dk, dv = torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda()
    binding.write_cache_fp8(w.k_new.cuda(), w.v_new.cuda(), w.slot_mapping.cuda(), dk, dv, k_scale, v_scale)
    out = binding.decode_fp8(w.q.cuda(), dk, dv, w.block_tables.cuda(), w.context_lens.cuda(), w.scale, k_scale,
                             v_scale)
    torch.cuda.synchronize()
    k_ref, v_ref = ofp8.write_cache_fp8(kcode, vcode, w.k_new.float().numpy(), w.v_new.float().numpy(),
                                        w.slot_mapping.numpy(), bs, k_scale, v_scale)
    assert np.array_equal(dk.cpu().numpy(), k_ref) and np.array_equal(dv.cpu().numpy(), v_ref)
    want = ofp8.decode_fp8(w.q.double().numpy(), k_ref, v_ref, w.block_tables.numpy(), w.context_lens.numpy(),
                           w.scale, bs, k_scale, v_scale)
    assert_close(out, want, "bf16", "fp8 step")


@pytest.mark.parametrize("name", ["llama3_8b", "long_split", "gqa8_d64", "llama_bs8", "llama_bs1", "llama_bs24"])
@pytest.mark.parametrize("num_ranges", [0, 997])
def test_fp8_append_equals_write_then_decode(name, num_ranges):
    """pa_decode_fp8_append: the newest tokens' quantising write fused into the
    decode gives the pools and output of pa_write_cache_fp8 + pa_decode_fp8."""
    sp = SMALL[name]
    w = workloads.make_workload(sp, prewritten=False)
    k_scale, v_scale = 0.37, 2.5
    kcode = _codes_of_pool(w, w.k_cache, k_scale)
    vcode = _codes_of_pool(w, w.v_cache, v_scale)
    bs = sp.block_size
    for s, c in enumerate(w.context_lens.tolist()):  # the newest slot holds poison until written
        if c > 0:
            slot = int(w.slot_mapping[s])
            kcode[slot // bs, slot % bs] = NAN_CODE
            vcode[slot // bs, slot % bs] = NAN_CODE
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    ka, va = torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda()
    binding.write_cache_fp8(kn, vn, w.slot_mapping.cuda(), ka, va, k_scale, v_scale)
    out_a = binding.decode_fp8(q, ka, va, bt, cl, w.scale, k_scale, v_scale, num_ranges=num_ranges)
    kb, vb = torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda()
    out_b = binding.decode_fp8_append(q, kn, vn, kb, vb, bt, cl, w.scale, k_scale, v_scale, num_ranges=num_ranges,
                                      check_block_ids=True)
    torch.cuda.synchronize()
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))


# ---- full size, in the launch form the benchmark times ----


def _compact(w, codes, seqs):
    """The sampled sequences' blocks of a code pool, relabelled 0.., with their
    tables, lengths and the local slot of each one's newest token."""
    bs = w.spec.block_size
    bt, ctx = w.block_tables.numpy(), w.context_lens.numpy()
    nblk = [-(-int(ctx[s]) // bs) for s in seqs]
    used = sorted({int(b) for s, n in zip(seqs, nblk) for b in bt[s, :n]})
    remap = {b: i for i, b in enumerate(used)}
    bt2 = np.full((len(seqs), max(nblk)), -1, dtype=np.int64)
    slots = np.full(len(seqs), -1, dtype=np.int64)
    for i, (s, n) in enumerate(zip(seqs, nblk)):
        bt2[i, :n] = [remap[int(b)] for b in bt[s, :n]]
        c = int(ctx[s])
        slots[i] = remap[int(bt[s, (c - 1) // bs])] * bs + (c - 1) % bs
    return codes[torch.as_tensor(used)].numpy(), bt2, ctx[seqs], slots


@pytest.mark.parametrize("name, sample", [("llama3_8b", [0, 7, 21, 40, 63]), ("long_ctx", [0, 3, 7])])
def test_full_size_fp8_append_sampled(name, sample):
    """pa_decode_fp8_append on the full batch: bit-identical to
    pa_write_cache_fp8 + pa_decode_fp8, the written codes equal the oracle's
    quantiser, and sampled sequences (the longest among them) match the oracle
    on the oracle-written pools.  The prompt's codes are torch's E4M3 cast of
    the pool over its scale (input generation)."""
    w = workloads.make_workload(name, prewritten=False)
    k_scale, v_scale = 0.37, 2.5
    kin = (w.k_cache.cuda().float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vin = (w.v_cache.cuda().float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    longest = int(torch.argmax(w.context_lens))
    sample = sorted(set(sample) | {longest})
    bs = w.spec.block_size
    used_ids = torch.as_tensor(sorted({int(b) for s in sample
                                       for b in w.block_tables[s, :-(-int(w.context_lens[s]) // bs)]}))
    k_before = torch.zeros_like(w.k_cache, dtype=torch.uint8)
    v_before = torch.zeros_like(w.v_cache, dtype=torch.uint8)
    k_before[used_ids] = kin[used_ids.cuda()].cpu()
    v_before[used_ids] = vin[used_ids.cuda()].cpu()
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    ka, va = kin.clone(), vin.clone()
    binding.write_cache_fp8(kn, vn, w.slot_mapping.cuda(), ka, va, k_scale, v_scale)
    out_a = binding.decode_fp8(q, ka, va, bt, cl, w.scale, k_scale, v_scale)
    out_b = binding.decode_fp8_append(q, kn, vn, kin, vin, bt, cl, w.scale, k_scale, v_scale)
    torch.cuda.synchronize()
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))
    assert torch.equal(kin, ka) and torch.equal(vin, va)
    del ka, va
    # The newest tokens' codes, against the oracle's quantiser.
    for s in sample:
        slot = int(w.slot_mapping[s])
        assert np.array_equal(kin[slot // bs, slot % bs].cpu().numpy(), ofp8.quantize(w.k_new[s].float().numpy(), k_scale))
        assert np.array_equal(vin[slot // bs, slot % bs].cpu().numpy(), ofp8.quantize(w.v_new[s].float().numpy(), v_scale))
    kc, bt2, ctx2, slots = _compact(w, k_before, sample)
    vc, _, _, _ = _compact(w, v_before, sample)
    k_ref, v_ref = ofp8.write_cache_fp8(kc, vc, w.k_new[sample].float().numpy(), w.v_new[sample].float().numpy(),
                                        slots, bs, k_scale, v_scale)
    want = ofp8.decode_fp8(w.q[sample].double().numpy(), k_ref, v_ref, bt2, ctx2, w.scale, bs, k_scale, v_scale)
    assert_close(out_b[sample], want, "bf16", f"fp8 full {name}")
    assert torch.isfinite(out_b).all()


# ---- several query tokens per sequence over FP8 pools ----

import oracle  # noqa: E402

MQ_CASES = {
    # (spec, Q): (query, head) columns per KV head 8 (one warp), 16, 12, 32, 24, 20
    "llama_q2": (SMALL["llama3_8b"], 2),
    "llama_q4": (SMALL["llama3_8b"], 4),
    "long_q3": (SMALL["long_split"], 3),
    "gqa8_q4": (SMALL["gqa8_bs32"], 4),
    "gqa8_d64_q3": (SMALL["gqa8_d64"], 3),
    "llama_bs24_q5": (SMALL["llama_bs24"], 5),
}


def _mq_queries(w, Q, seed):
    S, H, D = w.q.shape
    rng = np.random.default_rng([w.spec.seed, 79, Q, seed])
    return torch.from_numpy(rng.standard_normal((S, Q, H, D), dtype=np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("name", list(MQ_CASES))
@pytest.mark.parametrize("num_ranges", [0, 1, 5])
def test_fp8_multi_query_matches_oracle(name, num_ranges):
    sp, Q = MQ_CASES[name]
    w = workloads.make_workload(sp, prewritten=True)
    k_scale, v_scale = 0.5, 0.25
    kcode = _codes_of_pool(w, w.k_cache, k_scale)
    vcode = _codes_of_pool(w, w.v_cache, v_scale)
    q = _mq_queries(w, Q, 0)
    out = binding.decode_fp8_multi(q.cuda(), torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda(),
                                   w.block_tables.cuda(), w.context_lens.cuda(), w.scale, k_scale, v_scale,
                                   num_ranges=num_ranges)
    torch.cuda.synchronize()
    want = oracle.decode_multi(q.double().numpy(), ofp8.e4m3_decode(kcode) * k_scale,
                               ofp8.e4m3_decode(vcode) * v_scale, w.block_tables.numpy(), w.context_lens.numpy(),
                               w.scale, sp.block_size)
    assert_close(out, want, "bf16", f"fp8 mq {name} R={num_ranges}")


def test_fp8_multi_query_with_one_query_equals_fp8_decode():
    w = workloads.make_workload(SMALL["llama3_8b"], prewritten=True)
    kcode = torch.from_numpy(_codes_of_pool(w, w.k_cache, 0.5)).cuda()
    vcode = torch.from_numpy(_codes_of_pool(w, w.v_cache, 0.5)).cuda()
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    a = binding.decode_fp8_multi(w.q[:, None].contiguous().cuda(), kcode, vcode, bt, cl, w.scale, 0.5, 0.5)
    b = binding.decode_fp8(w.q.cuda(), kcode, vcode, bt, cl, w.scale, 0.5, 0.5)
    torch.cuda.synchronize()
    assert torch.equal(a[:, 0], b)


@pytest.mark.parametrize("name", ["llama_q2", "llama_q4", "gqa8_q4", "gqa8_d64_q3", "llama_bs24_q5"])
@pytest.mark.parametrize("num_ranges", [0, 997])
def test_fp8_mq_append_equals_write_then_decode(name, num_ranges):
    """pa_decode_fp8_mq_append: the Q new rows' quantising write fused into the
    decode (one launch up to 8 columns per KV head, a row-writing kernel
    chained ahead above that) gives the pools and output of
    pa_write_cache_fp8 + pa_decode_fp8_mq bit for bit."""
    sp, Q = MQ_CASES[name]
    w = workloads.make_workload(sp, prewritten=True)
    k_scale, v_scale = 0.37, 2.5
    kcode = _codes_of_pool(w, w.k_cache, k_scale)
    vcode = _codes_of_pool(w, w.v_cache, v_scale)
    S = sp.num_seqs
    bs = sp.block_size
    rng = np.random.default_rng([sp.seed, 80, Q])
    Hk, D = w.k_cache.shape[2], w.k_cache.shape[3]
    kn = torch.from_numpy(rng.standard_normal((S * Q, Hk, D), dtype=np.float32) * 2).to(torch.bfloat16)
    vn = torch.from_numpy(rng.standard_normal((S * Q, Hk, D), dtype=np.float32) * 2).to(torch.bfloat16)
    slots = np.full(S * Q, -1, dtype=np.int64)
    for s, c in enumerate(w.context_lens.tolist()):
        for i in range(Q):
            pos = c - Q + i
            if pos >= 0:
                slots[s * Q + i] = int(w.block_tables[s, pos // bs]) * bs + pos % bs
                kcode[slots[s * Q + i] // bs, slots[s * Q + i] % bs] = NAN_CODE  # poison until written
                vcode[slots[s * Q + i] // bs, slots[s * Q + i] % bs] = NAN_CODE
    q = _mq_queries(w, Q, 1).cuda()
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    ka, va = torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda()
    binding.write_cache_fp8(kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda(), ka, va, k_scale, v_scale)
    out_a = binding.decode_fp8_multi(q, ka, va, bt, cl, w.scale, k_scale, v_scale, num_ranges=num_ranges)
    kb, vb = torch.from_numpy(kcode).cuda(), torch.from_numpy(vcode).cuda()
    out_b = binding.decode_fp8_multi_append(q, kn.cuda(), vn.cuda(), kb, vb, bt, cl, w.scale, k_scale, v_scale,
                                            num_ranges=num_ranges, check_block_ids=True)
    torch.cuda.synchronize()
    assert torch.equal(kb, ka) and torch.equal(vb, va)
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))
    # The written codes are the oracle quantiser's.
    k_ref, v_ref = ofp8.write_cache_fp8(kcode, vcode, kn.float().numpy(), vn.float().numpy(), slots, bs, k_scale,
                                        v_scale)
    assert np.array_equal(kb.cpu().numpy(), k_ref) and np.array_equal(vb.cpu().numpy(), v_ref)
    want = oracle.decode_multi(q.double().cpu().numpy(), ofp8.e4m3_decode(k_ref) * k_scale,
                               ofp8.e4m3_decode(v_ref) * v_scale, w.block_tables.numpy(), w.context_lens.numpy(),
                               w.scale, bs)
    assert_close(out_b, want, "bf16", f"fp8 mq append {name}")
