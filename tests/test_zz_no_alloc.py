"""pa_decode_static: the decode entry point that allocates nothing.

Callers that cannot call cudaMalloc when they decode (an engine whose allocator
already holds nearly all device memory, or a path that cannot take
cudaMalloc's implicit device synchronisation) use this entry point; its
scratch is an array compiled into the library.  These tests call it through
the C ABI and check it against pa_decode on the same inputs, twice in a row,
since every call reuses the same array.  The file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import TOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_292_gb300 import build

    build.build()
    return binding.load()


def _call(fn, out, w, g, stream):
    sp = w.spec
    S, H, D = w.q.shape
    return fn(out.data_ptr(), g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
              g["block_tables"].data_ptr(), g["context_lens"].data_ptr(), S, H, sp.num_kv_heads, D,
              sp.block_size, w.max_blocks_per_seq, w.scale, stream, binding.dtype_code(w.q.dtype))


def _assert_close(got, ref, dtype):
    err = (got.double() - ref.double()).abs()
    max_tol, mean_tol = TOL[dtype]
    assert torch.isfinite(got).all()
    assert err.max().item() <= max_tol
    if mean_tol is not None:
        assert err.mean().item() <= mean_tol


@pytest.mark.parametrize(
    "sp",
    [
        workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600),
        workloads.spec("long_ctx", num_seqs=2, ctx_lo=3001, ctx_hi=3001, max_context=3008, pool_blocks=0),
        workloads.spec("tiny_fp32"),
    ],
    ids=["llama-shaped", "long-split", "tiny-fp32"],
)
def test_static_matches_pa_decode_twice(lib, sp):
    w = workloads.make_workload(sp, prewritten=True, poison=True)
    g = to_device(w)
    stream = torch.cuda.current_stream().cuda_stream
    ref = torch.empty_like(g["q"])
    assert _call(lib.pa_decode, ref, w, g, stream) == binding.PA_OK
    for _ in range(2):
        out = torch.full_like(g["q"], float("nan"))
        rc = _call(lib.pa_decode_static, out, w, g, stream)
        assert rc == binding.PA_OK, lib.pa_last_error()
        torch.cuda.synchronize()
        _assert_close(out, ref, sp.dtype)


def test_static_rejects_oversized_batches(lib):
    # A million sequences: their merge tickets alone exceed the compiled-in array.
    need = lib.pa_decode_workspace_size(1_000_000, 32, 8, 128, 0)
    assert need > 16 * 1024 * 1024
    rc = lib.pa_decode_static(16, 16, 16, 16, 16, 16, 1_000_000, 32, 8, 128, 16, 8, 0.1, 0, binding.PA_BF16)
    assert rc == binding.PA_ERR_WORKSPACE
    assert b"scratch" in ctypes.string_at(lib.pa_last_error())
