"""Steady-state decode: the host block manager, the copy-on-write block copy,
the cache write and paged decode driven together for several steps.

Each sequence's K/V history is kept on the host as the ground truth; every
step's decode output is compared with the fp64 oracle's attention over that
history.  Forks (shared blocks that later diverge), a shared prefix, and a
freed sequence whose blocks are reused are all exercised; the pool starts
filled with NaN so any read of a slot no token owns shows up."""

import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_292_gb300 import binding

from paritylib import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


class _Loop:
    def __init__(self, nb, bs, seqs, mb, H, Hk, D, dtype, seed):
        self.bm = binding.BlockManager(nb, bs, seqs, mb)
        self.nb, self.bs, self.H, self.Hk, self.D, self.dtype = nb, bs, H, Hk, D, dtype
        self.k = torch.full((nb, bs, Hk, D), float("nan"), dtype=dtype, device="cuda")
        self.v = torch.full_like(self.k, float("nan"))
        self.hist_k = [[] for _ in range(seqs)]
        self.hist_v = [[] for _ in range(seqs)]
        self.gen = torch.Generator().manual_seed(seed)
        self.copies = 0

    def add_tokens(self, seq, n):
        slots, copies = self.bm.append(seq, n)
        if copies:
            pairs = torch.tensor(copies, dtype=torch.int32, device="cuda")
            binding.pa_copy_blocks(self.k, self.v, pairs, len(copies), self.Hk, self.D, self.bs, self.nb)
            self.copies += len(copies)
        kn = torch.randn(n, self.Hk, self.D, generator=self.gen).to(self.dtype)
        vn = torch.randn(n, self.Hk, self.D, generator=self.gen).to(self.dtype)
        binding.write_cache(kn.cuda(), vn.cuda(), slots.cuda(), self.k, self.v)
        self.hist_k[seq].extend(kn)
        self.hist_v[seq].extend(vn)

    def fork(self, parent, child):
        self.bm.fork(parent, child)
        self.hist_k[child] = list(self.hist_k[parent])
        self.hist_v[child] = list(self.hist_v[parent])

    def share_prefix(self, seq, donor, n):
        self.bm.share_prefix(seq, donor, n)
        self.hist_k[seq] = list(self.hist_k[donor][:n])
        self.hist_v[seq] = list(self.hist_v[donor][:n])

    def free(self, seq):
        self.bm.free(seq)
        self.hist_k[seq], self.hist_v[seq] = [], []

    def decode_and_check(self, step):
        tables, lens = self.bm.export()
        S = tables.shape[0]
        q = torch.randn(S, self.H, self.D, generator=self.gen).to(self.dtype)
        scale = 1 / math.sqrt(self.D)
        out = binding.decode(q.cuda(), self.k, self.v, tables.cuda(), lens.cuda(), scale, check_block_ids=True)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        for s in range(S):
            if not self.hist_k[s]:
                assert np.all(got[s] == 0)
                continue
            ks = torch.stack(self.hist_k[s]).double().numpy()
            vs = torch.stack(self.hist_v[s]).double().numpy()
            want = oracle.attention(q[s].double().numpy(), ks, vs, scale)
            # max-abs and (bf16) mean-abs bounds, per sequence and step
            assert_close(out[s], want, "f32" if self.dtype == torch.float32 else "bf16", f"step {step} seq {s}")


@pytest.mark.parametrize("dtype, D, bs", [(torch.bfloat16, 128, 16), (torch.float32, 64, 8), (torch.bfloat16, 64, 32)])
def test_multistep_decode_with_forks_prefix_and_reuse(dtype, D, bs):
    rng = np.random.default_rng(11)
    loop = _Loop(nb=400, bs=bs, seqs=8, mb=48, H=16, Hk=4, D=D, dtype=dtype, seed=5)
    for s in range(5):
        loop.add_tokens(s, int(rng.integers(1, 150)))
    loop.fork(0, 5)  # beam-style fork: shares every block, including a partial last one
    donor_len = loop.bm.context_len(1)
    loop.share_prefix(6, 1, (donor_len // bs) * bs)  # prefix cache hit on whole blocks
    loop.add_tokens(6, 3)
    loop.decode_and_check(-1)
    for step in range(6):
        for s in range(8):
            if loop.bm.context_len(s) > 0:
                loop.add_tokens(s, 1)
        if step == 2:
            loop.free(3)  # its blocks go back to the pool and are reused next
            loop.add_tokens(7, 40)
        loop.decode_and_check(step)
    assert loop.copies >= 1  # the fork forced at least one copy-on-write
    loop.bm.close()


def test_copy_blocks_is_a_bit_copy():
    nb, bs, hk, d = 12, 16, 8, 128
    k = torch.randn(nb, bs, hk, d).to(torch.bfloat16).cuda()
    v = torch.randn(nb, bs, hk, d).to(torch.bfloat16).cuda()
    k0, v0 = k.clone(), v.clone()
    pairs = torch.tensor([[3, 7], [1, 0], [11, 4]], dtype=torch.int32, device="cuda")
    binding.pa_copy_blocks(k, v, pairs, 3, hk, d, bs, nb)
    torch.cuda.synchronize()
    want_k, want_v = k0.clone(), v0.clone()
    for src, dst in pairs.tolist():
        want_k[dst], want_v[dst] = k0[src], v0[src]
    assert torch.equal(k.view(torch.int16), want_k.view(torch.int16))
    assert torch.equal(v.view(torch.int16), want_v.view(torch.int16))
