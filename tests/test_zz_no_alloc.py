"""pa_decode_static: the decode entry point that allocates nothing.

Some callers cannot call cudaMalloc when they decode: an engine whose own
allocator already holds nearly all device memory, or a path that cannot take
cudaMalloc's implicit device synchronisation.  They use this entry point,
whose scratch is an array compiled into the library.  These tests call it
through the C ABI and compare it with pa_decode on the same inputs, several
calls in a row, since every call reuses the one array.  The file is collected
last on purpose.
"""

import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from paged_kv_cache_292_gb300 import binding, workloads

from paritylib import TOL, to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
        # Same launch plan as pa_decode, so the very same bits.
        assert torch.equal(out, ref)


# Run in a fresh process, where nothing has touched the library before: only
# pa_decode_static is called at first, and the device's free memory must not
# move.  The library carries its own CUDA runtime, which loads all of the
# library's modules (the scratch array with them) on its first call when
# CUDA_MODULE_LOADING=EAGER; one pa_write_cache call of a padding token (it
# allocates nothing) makes that happen before the first reading, so a later
# change can only come from an allocation.  The long-context
# batch runs first: its partial results land where the fp32 batch keeps its
# merge tickets in the shared array, so the fp32 calls are correct only if
# each call clears its tickets.  pa_decode (which may allocate) runs last and
# must give the same bits.
_CHILD = textwrap.dedent(
    r"""
    import sys
    sys.path.insert(0, sys.argv[1])
    sys.path.insert(0, sys.argv[1] + "/tests")
    import torch
    from paged_kv_cache_292_gb300 import binding, workloads
    from paritylib import to_device

    lib = binding.load()
    torch.cuda.init()
    specs = [
        workloads.spec("long_ctx", num_seqs=2, ctx_lo=3001, ctx_hi=3001, max_context=3008, pool_blocks=0),
        workloads.spec("tiny_fp32"),
        workloads.spec("tiny_fp32"),
        workloads.spec("llama3_8b", num_seqs=12, ctx_lo=1, ctx_hi=700, max_context=704, pool_blocks=600),
    ]
    cases = []
    for sp in specs:
        w = workloads.make_workload(sp, prewritten=True, poison=True)
        g = to_device(w)
        out = torch.full(tuple(w.q.shape), float("nan"), dtype=w.q.dtype).cuda()
        cases.append((w, g, out))
    torch.cuda.synchronize()

    def call(fn, w, g, out):
        S, H, D = w.q.shape
        return fn(out.data_ptr(), g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
                  g["block_tables"].data_ptr(), g["context_lens"].data_ptr(), S, H, w.spec.num_kv_heads, D,
                  w.spec.block_size, w.max_blocks_per_seq, w.scale, 0, binding.dtype_code(w.q.dtype))

    w0, g0, _ = cases[1]
    pad = torch.full((1,), -1, dtype=torch.int64).cuda()
    _, Hk0, D0 = w0.k_new.shape
    assert lib.pa_write_cache(g0["k_new"].data_ptr(), g0["v_new"].data_ptr(), pad.data_ptr(),
                              g0["k_cache"].data_ptr(), g0["v_cache"].data_ptr(), 1, Hk0, D0,
                              w0.spec.block_size, w0.num_blocks, 0, binding.dtype_code(w0.k_new.dtype)) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for w, g, out in cases:
        rc = call(lib.pa_decode_static, w, g, out)
        assert rc == 0, lib.pa_last_error()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert free1 == free0, ("device memory moved", free0, free1)
    for i, (w, g, out) in enumerate(cases):
        ref = torch.empty_like(out)
        assert call(lib.pa_decode, w, g, ref) == 0, lib.pa_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out, ref), ("differs from pa_decode", i)
    print("no-alloc ok")
    """
)


def test_static_in_fresh_process_allocates_nothing_and_clears_tickets(lib):
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "no-alloc ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_static_rejects_oversized_batches(lib):
    # A million sequences: their merge tickets alone exceed the compiled-in array.
    need = lib.pa_decode_workspace_size(1_000_000, 32, 8, 128, 0)
    assert need > 16 * 1024 * 1024
    rc = lib.pa_decode_static(16, 16, 16, 16, 16, 16, 1_000_000, 32, 8, 128, 16, 8, 0.1, 0, binding.PA_BF16)
    assert rc == binding.PA_ERR_WORKSPACE
    assert b"scratch" in ctypes.string_at(lib.pa_last_error())
