"""The decode step captured into a CUDA graph, in both launch forms (cache
write + pa_decode_ws, and the fused pa_decode_append with caller scratch):
replays give the same result as eager calls and as the oracle.  With caller
scratch neither allocates nor synchronises, so both can be captured."""

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


@pytest.mark.parametrize("name", ["llama3_8b", "tiny_fp32"])
def test_captured_step_matches_eager_and_oracle(name):
    if name == "llama3_8b":
        sp = workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600)
    else:
        sp = workloads.spec("tiny_fp32")
    w = workloads.make_workload(sp, prewritten=False, poison=True)
    g = to_device(w)
    S, H, D = w.q.shape
    Hk, bs, NB, MB = sp.num_kv_heads, sp.block_size, w.num_blocks, w.max_blocks_per_seq
    need = binding.pa_decode_workspace_size(S, H, Hk, D)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(g["q"])

    def step():
        binding.pa_write_cache(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"], S, Hk, D, bs, NB)
        binding.pa_decode_ws(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"], S, H, Hk,
                             D, bs, MB, w.scale, None, None, ws, need)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    k_ref, v_ref = oracle_pools_after_write(w)
    assert_close(out, oracle_decode(w, k_ref, v_ref), sp.dtype, f"graph {name}")


def test_captured_fused_step_matches_eager_and_oracle():
    """The step the benchmark times, pa_decode_append with caller scratch,
    captured once and replayed: each replay writes the newest tokens again
    (the same bytes) and decodes."""
    sp = workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600)
    w = workloads.make_workload(sp, prewritten=False, poison=True)
    g = to_device(w)
    S, H, D = w.q.shape
    need = binding.pa_decode_workspace_size(S, H, sp.num_kv_heads, D)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(g["q"])

    def step():
        binding.decode_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], w.scale, out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    k_ref, v_ref = oracle_pools_after_write(w)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), k_ref.view(torch.int16))
    assert_close(out, oracle_decode(w, k_ref, v_ref), "bf16", "graph fused step")
