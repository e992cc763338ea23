"""The decode pipeline's bounded waits, driven to run out without any fault.

Every wait in the decode kernel gives up after a time limit, reports
PA_DEVERR_TIMEOUT and ends the kernel early, so that a copy that never lands
cannot hang the GPU.  pa_test_stall_copy makes the next launch withhold one
tile's copies (that stage's barrier is never armed, so nothing ever completes
it) and bounds every wait by 1 ms.  Each test checks that the call returns
within a fraction of a second, that the error word carries the timeout bit,
and that the context and the scratch (zero-filled again, as after any timeout)
serve the next call, whose output equals the one taken before the stall.
"""

import time

import numpy as np
import pytest
import torch

from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    binding.load()


def _total_tiles(w):
    return int(sum(-(-int(c) // 16) for c in w.context_lens.tolist()))


def _run(kind, w, g, ws, flag, queries=None):
    if kind == "fp8":
        return binding.decode_fp8(g["q"], g["k8"], g["v8"], g["block_tables"], g["context_lens"], w.scale, 0.5,
                                  0.5, workspace=ws, error_flag=flag)
    if kind == "mq":
        return binding.decode_multi(queries, g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"],
                                    w.scale, workspace=ws, error_flag=flag)
    return binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                          workspace=ws, error_flag=flag)


@pytest.mark.parametrize("kind", ["bf16", "f32", "fp8", "mq"])
@pytest.mark.parametrize("where", [0.0, 0.5, 1.0])
def test_withheld_copy_times_out_and_the_next_call_is_clean(kind, where):
    if kind == "f32":
        sp = workloads.spec("tiny_fp32")
    else:
        sp = workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600)
    w = workloads.make_workload(sp, prewritten=True)
    g = to_device(w)
    S, H, D = w.q.shape
    Hk = sp.num_kv_heads
    queries = None
    if kind == "fp8":
        g["k8"] = (g["k_cache"].float() / 0.5).to(torch.float8_e4m3fn).view(torch.uint8)
        g["v8"] = (g["v_cache"].float() / 0.5).to(torch.float8_e4m3fn).view(torch.uint8)
        need = binding.pa_decode_workspace_size(S, H, Hk, D)
    elif kind == "mq":
        gen = torch.Generator().manual_seed(3)
        queries = torch.randn(S, 4, H, D, generator=gen).to(torch.bfloat16).cuda()  # G * Q = 16: two warps per KV head
        need = binding.pa_decode_mq_workspace_size(S, 4, H, Hk, D)
    else:
        need = binding.pa_decode_workspace_size(S, H, Hk, D)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _run(kind, w, g, ws, flag, queries).clone()
    torch.cuda.synchronize()
    assert int(flag.item()) == 0

    tile = min(int(where * _total_tiles(w)), _total_tiles(w) - 1)
    binding.pa_test_stall_copy(tile, 1000)
    t0 = time.perf_counter()
    _run(kind, w, g, ws, flag, queries)
    torch.cuda.synchronize()
    took = time.perf_counter() - t0
    assert int(flag.item()) & binding.PA_DEVERR_TIMEOUT
    assert took < 0.5, took  # a few 1 ms limits, not the default 2 s

    # The setting was used once; the scratch is zeroed as after any timeout.
    ws.zero_()
    flag.zero_()
    out = _run(kind, w, g, ws, flag, queries)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert torch.equal(out, ref)
    tickets = (4 * S * Hk + 255) // 256 * 256  # the merge tickets occupy the scratch's last bytes
    assert int(ws[need - tickets:].view(torch.int32).abs().sum()) == 0


def test_stall_of_a_tile_past_the_batch_changes_nothing():
    """A tile index no range owns: nothing is withheld and nothing times out."""
    w = workloads.make_workload("tiny_fp32", prewritten=True)
    g = to_device(w)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale)
    binding.pa_test_stall_copy(10 ** 9, 1000)
    out = binding.decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], w.scale,
                         error_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert torch.equal(out, ref)
    assert np.isfinite(out.cpu().numpy()).all()
