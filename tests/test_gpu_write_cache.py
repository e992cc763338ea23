"""GPU parity of the cache write (reshape-and-cache scatter): bit-exact."""

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import int_view

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


def _rand_case(dtype, nb, bs, hk, d, slots, seed=0):
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    kc = torch.randn(nb, bs, hk, d, generator=g).to(tdt)
    vc = torch.randn(nb, bs, hk, d, generator=g).to(tdt)
    t = len(slots)
    kn = torch.randn(t, hk, d, generator=g).to(tdt)
    vn = torch.randn(t, hk, d, generator=g).to(tdt)
    return kc, vc, kn, vn, torch.tensor(slots, dtype=torch.int64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("hk, d, bs", [(8, 128, 16), (8, 64, 32), (1, 64, 16), (16, 128, 8), (2, 128, 1)])
def test_write_cache_bit_exact(dtype, hk, d, bs):
    nb = 37
    rng = np.random.default_rng(hk * 1000 + d + bs)
    slots = rng.choice(nb * bs, size=min(50, nb * bs), replace=False).tolist()
    slots[3] = -1  # padding token
    slots[7] = -5
    kc, vc, kn, vn, sm = _rand_case(dtype, nb, bs, hk, d, slots)
    view = int_view(dtype)
    k_ref, v_ref = oracle.write_cache(kc.view(view).numpy(), vc.view(view).numpy(), kn.view(view).numpy(),
                                      vn.view(view).numpy(), sm.numpy(), bs)
    dk, dv = kc.cuda(), vc.cuda()
    binding.write_cache(kn.cuda(), vn.cuda(), sm.cuda(), dk, dv)
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().view(view).numpy(), k_ref)
    assert np.array_equal(dv.cpu().view(view).numpy(), v_ref)


def test_out_of_pool_slot_is_skipped_and_reported():
    nb, bs = 5, 16
    kc, vc, kn, vn, sm = _rand_case("bf16", nb, bs, 8, 128, [3, nb * bs, 17, nb * bs + 1000])
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    dk, dv = kc.cuda(), vc.cuda()
    binding.write_cache(kn.cuda(), vn.cuda(), sm.cuda(), dk, dv, error_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & binding.PA_DEVERR_SLOT
    valid = torch.tensor([3, -1, 17, -1], dtype=torch.int64)
    k_ref, _ = oracle.write_cache(kc.view(torch.int16).numpy(), vc.view(torch.int16).numpy(),
                                  kn.view(torch.int16).numpy(), vn.view(torch.int16).numpy(), valid.numpy(), bs)
    assert np.array_equal(dk.cpu().view(torch.int16).numpy(), k_ref)


def test_zero_tokens_is_a_no_op():
    kc, vc, kn, vn, sm = _rand_case("bf16", 4, 16, 8, 128, [])
    dk = kc.cuda()
    binding.write_cache(kn.reshape(0, 8, 128).cuda(), vn.reshape(0, 8, 128).cuda(), sm.cuda(), dk, vc.cuda())
    torch.cuda.synchronize()
    assert torch.equal(dk.cpu().view(torch.int16), kc.view(torch.int16))


def test_workload_step_write_matches_generator_layout():
    """Writing the step's new tokens into the unwritten pool reproduces the
    generator's pre-written pool bit for bit (llama-shaped, full pool)."""
    post = workloads.make_workload("llama3_8b", prewritten=False)
    pre_k = workloads.make_workload("llama3_8b", prewritten=True).k_cache
    dk, dv = post.k_cache.cuda(), post.v_cache.cuda()
    binding.write_cache(post.k_new.cuda(), post.v_new.cuda(), post.slot_mapping.cuda(), dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(dk.view(torch.int16), pre_k.cuda().view(torch.int16))
