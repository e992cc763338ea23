"""Full-size parity of the multi-query steps the benchmark times.

The batches are the benchmark's own (bench.py --queries Q, with --kv fp8 for
the FP8 pool): the full Llama-3-8B-shaped and 70B-shaped workloads with Q new
tokens per sequence at positions ctx - Q .. ctx - 1 (workloads.multi_query_step).
For each, the fused call the benchmark times (pa_decode_mq_append /
pa_decode_fp8_mq_append) must give the same output and pools, bit for bit, as
the cache write followed by the decode; sampled sequences (the longest always
among them) must match the fp64 oracle run on the oracle-written pools.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8 as ofp8
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


def _compact(w, seqs, slots, Q):
    """The listed sequences' blocks, relabelled 0.. in order of block id: the
    block ids, the relabelled tables and lengths, and the relabelled slots of
    the sequences' Q new rows (rows s * Q .. s * Q + Q - 1; -1 stays -1)."""
    bs = w.spec.block_size
    bt, ctx = w.block_tables.numpy(), w.context_lens.numpy()
    nblk = [-(-int(ctx[s]) // bs) for s in seqs]
    used = sorted({int(b) for s, n in zip(seqs, nblk) for b in bt[s, :n]})
    remap = {b: i for i, b in enumerate(used)}
    bt2 = np.full((len(seqs), max(nblk)), -1, dtype=np.int64)
    for i, (s, n) in enumerate(zip(seqs, nblk)):
        bt2[i, :n] = [remap[int(b)] for b in bt[s, :n]]
    rows = [s * Q + j for s in seqs for j in range(Q)]
    sl = slots.numpy()[rows]
    sl2 = np.array([-1 if x < 0 else remap[int(x) // bs] * bs + int(x) % bs for x in sl], dtype=np.int64)
    return torch.as_tensor(used), bt2, ctx[seqs], rows, sl2


FULL_MQ = [("llama3_8b", 2, [0, 7, 21, 40, 63]), ("llama3_8b", 4, [0, 7, 21, 40, 63]),
           ("gqa8_70b", 2, [0, 31, 64, 127]), ("gqa8_70b", 4, [3, 64, 100])]


@pytest.mark.parametrize("name, Q, sample", FULL_MQ)
def test_full_size_mq_append_sampled(name, Q, sample):
    w = workloads.make_workload(name, prewritten=False)
    q, kn, vn, slots = workloads.multi_query_step(w, Q)
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
    kf, vf = w.k_cache.cuda(), w.v_cache.cuda()
    out_f = binding.decode_multi_append(qd, knd, vnd, kf, vf, bt, cl, w.scale, check_block_ids=True)
    ka, va = w.k_cache.cuda(), w.v_cache.cuda()
    binding.write_cache(knd, vnd, slots.cuda(), ka, va)
    out_a = binding.decode_multi(qd, ka, va, bt, cl, w.scale)
    torch.cuda.synchronize()
    i16 = torch.int16
    assert torch.equal(out_f.view(i16), out_a.view(i16))
    assert torch.equal(kf.view(i16), ka.view(i16)) and torch.equal(vf.view(i16), va.view(i16))
    del ka, va
    assert torch.isfinite(out_f).all()
    longest = int(torch.argmax(w.context_lens))
    sample = sorted(set(sample) | {longest})
    used, bt2, ctx2, rows, sl2 = _compact(w, sample, slots, Q)
    # Written rows are the new tokens, bit for bit.
    bs = w.spec.block_size
    for r in rows:
        x = int(slots[r])
        if x >= 0:
            assert torch.equal(kf[x // bs, x % bs].cpu().view(i16), kn[r].view(i16))
            assert torch.equal(vf[x // bs, x % bs].cpu().view(i16), vn[r].view(i16))
    del kf, vf
    k2, v2 = oracle.write_cache(w.k_cache[used].view(i16).numpy(), w.v_cache[used].view(i16).numpy(),
                                kn[rows].view(i16).numpy(), vn[rows].view(i16).numpy(), sl2, bs)
    kd = torch.from_numpy(k2).view(torch.bfloat16).double().numpy()
    vd = torch.from_numpy(v2).view(torch.bfloat16).double().numpy()
    want = oracle.decode_multi(q[sample].double().numpy(), kd, vd, bt2, ctx2, w.scale, bs)
    assert_close(out_f[sample], want, "bf16", f"full {name} Q={Q}")


@pytest.mark.parametrize("Q, sample", [(2, [0, 7, 21, 40, 63]), (4, [0, 7, 21, 40, 63])])
def test_full_size_fp8_mq_append_sampled(Q, sample):
    """FP8 pools (scales 1, as the benchmark): the prompt's codes are torch's
    E4M3 cast of the generator's pool (input generation); the fused call's new
    codes equal the oracle quantiser's."""
    w = workloads.make_workload("llama3_8b", prewritten=False)
    k_scale = v_scale = 1.0
    kin = (w.k_cache.cuda().float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vin = (w.v_cache.cuda().float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    q, kn, vn, slots = workloads.multi_query_step(w, Q)
    bt, cl = w.block_tables.cuda(), w.context_lens.cuda()
    qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
    longest = int(torch.argmax(w.context_lens))
    sample = sorted(set(sample) | {longest})
    used, bt2, ctx2, rows, sl2 = _compact(w, sample, slots, Q)
    k_before, v_before = kin[used.cuda()].cpu().numpy(), vin[used.cuda()].cpu().numpy()
    ka, va = kin.clone(), vin.clone()
    binding.write_cache_fp8(knd, vnd, slots.cuda(), ka, va, k_scale, v_scale)
    out_a = binding.decode_fp8_multi(qd, ka, va, bt, cl, w.scale, k_scale, v_scale)
    out_b = binding.decode_fp8_multi_append(qd, knd, vnd, kin, vin, bt, cl, w.scale, k_scale, v_scale,
                                            check_block_ids=True)
    torch.cuda.synchronize()
    assert torch.equal(out_b.view(torch.int16), out_a.view(torch.int16))
    assert torch.equal(kin, ka) and torch.equal(vin, va)
    del ka, va
    assert torch.isfinite(out_b).all()
    bs = w.spec.block_size
    for r in rows:
        x = int(slots[r])
        if x >= 0:
            assert np.array_equal(kin[x // bs, x % bs].cpu().numpy(), ofp8.quantize(kn[r].float().numpy(), k_scale))
            assert np.array_equal(vin[x // bs, x % bs].cpu().numpy(), ofp8.quantize(vn[r].float().numpy(), v_scale))
    k_ref, v_ref = ofp8.write_cache_fp8(k_before, v_before, kn[rows].float().numpy(), vn[rows].float().numpy(), sl2,
                                        bs, k_scale, v_scale)
    want = oracle.decode_multi(q[sample].double().numpy(), ofp8.e4m3_decode(k_ref) * k_scale,
                               ofp8.e4m3_decode(v_ref) * v_scale, bt2, ctx2, w.scale, bs)
    assert_close(out_b[sample], want, "bf16", f"fp8 full Q={Q}")
