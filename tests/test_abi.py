"""C-ABI library: builds, loads, exports the header's symbols, rejects bad
arguments on the host (no GPU and no kernel launch needed)."""

import ctypes
import os
import subprocess

import pytest

from paged_kv_cache_292_gb300 import binding
from paged_kv_cache_292_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return binding.load()


def test_library_exports_every_header_symbol(lib):
    names = binding.header_symbols()
    assert {"pa_decode", "pa_decode_ws", "pa_decode_ex", "pa_decode_workspace_size", "pa_write_cache",
            "pa_write_cache_ex", "pa_last_error", "pa_version"} <= set(names)
    raw = ctypes.CDLL(binding.library_path())
    for n in names:
        assert hasattr(raw, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()], capture_output=True, text=True)
    exported = {line.split()[-1] for line in nm.stdout.splitlines() if " T " in line}
    assert set(names) <= exported
    # ...and nothing else of the library's own: every exported pa_* symbol is
    # declared (and documented) in a header.
    assert {n for n in exported if n.startswith("pa_")} == set(names)
    assert lib.pa_version() == 100


def _decode_args(**kw):
    a = dict(out=16, query=16, k_cache=16, v_cache=16, block_tables=16, context_lens=16, num_seqs=1, num_heads=8,
             num_kv_heads=8, head_size=128, block_size=16, max_blocks_per_seq=4, scale=0.1, stream=0,
             dtype=binding.PA_BF16)
    a.update(kw)
    return a


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(out=None), binding.PA_ERR_INVALID_ARG),
        (dict(block_tables=None), binding.PA_ERR_INVALID_ARG),
        (dict(num_seqs=0), binding.PA_ERR_INVALID_ARG),
        (dict(num_heads=12, num_kv_heads=8), binding.PA_ERR_INVALID_ARG),
        (dict(num_heads=72, num_kv_heads=4), binding.PA_ERR_UNSUPPORTED),  # group 18 > 8
        (dict(head_size=96), binding.PA_ERR_UNSUPPORTED),
        (dict(dtype=7), binding.PA_ERR_UNSUPPORTED),
        (dict(block_size=0), binding.PA_ERR_INVALID_ARG),
        (dict(out=18), binding.PA_ERR_INVALID_ARG),  # misaligned
        (dict(scale=float("nan")), binding.PA_ERR_INVALID_ARG),
        (dict(head_size=256), binding.PA_ERR_UNSUPPORTED),
    ],
)
@pytest.mark.parametrize("entry", ["pa_decode", "pa_decode_static"])
def test_decode_rejects_bad_arguments_on_host(lib, kw, code, entry):
    """pa_decode_static checks its arguments as pa_decode does, with the same codes."""
    a = _decode_args(**kw)
    rc = getattr(lib, entry)(a["out"], a["query"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"],
                       a["num_seqs"], a["num_heads"], a["num_kv_heads"], a["head_size"], a["block_size"],
                       a["max_blocks_per_seq"], a["scale"], a["stream"], a["dtype"])
    assert rc == code
    assert lib.pa_last_error().decode()


def test_decode_ws_requires_workspace(lib):
    a = _decode_args()
    rc = lib.pa_decode_ws(a["out"], a["query"], a["k_cache"], a["v_cache"], a["block_tables"], a["context_lens"],
                          1, 8, 8, 128, 16, 4, 0.1, 0, binding.PA_BF16, None, 0)
    assert rc == binding.PA_ERR_INVALID_ARG


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(k_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(num_physical_blocks=0), binding.PA_ERR_INVALID_ARG),
        (dict(dtype=3), binding.PA_ERR_UNSUPPORTED),
        (dict(head_size=3, num_kv_heads=1), binding.PA_ERR_UNSUPPORTED),  # 6-byte rows
        (dict(k_cache=24), binding.PA_ERR_INVALID_ARG),
    ],
)
def test_write_cache_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(k_new=16, v_new=16, slot_mapping=16, k_cache=16, v_cache=16, num_tokens=4, num_kv_heads=8,
             head_size=128, block_size=16, num_physical_blocks=10, stream=0, dtype=binding.PA_BF16)
    a.update(kw)
    rc = lib.pa_write_cache(a["k_new"], a["v_new"], a["slot_mapping"], a["k_cache"], a["v_cache"], a["num_tokens"],
                            a["num_kv_heads"], a["head_size"], a["block_size"], a["num_physical_blocks"],
                            a["stream"], a["dtype"])
    assert rc == code


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(k_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(v_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(k_new=24), binding.PA_ERR_INVALID_ARG),  # misaligned
        (dict(dtype=binding.PA_F32), binding.PA_ERR_UNSUPPORTED),
        (dict(block_tables=None), binding.PA_ERR_INVALID_ARG),
    ],
)
def test_decode_append_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(out=16, query=16, k_new=16, v_new=16, k_cache=16, v_cache=16, block_tables=16, context_lens=16,
             dtype=binding.PA_BF16)
    a.update(kw)
    rc = lib.pa_decode_append(a["out"], a["query"], a["k_new"], a["v_new"], a["k_cache"], a["v_cache"],
                              a["block_tables"], a["context_lens"], 1, 8, 8, 128, 16, 4, 0.1, 0, a["dtype"], 0,
                              None, 0, 0, None)
    assert rc == code
    assert lib.pa_last_error().decode()


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(k_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(k_scale=0.0), binding.PA_ERR_INVALID_ARG),
        (dict(v_scale=float("inf")), binding.PA_ERR_INVALID_ARG),
    ],
)
def test_decode_fp8_append_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(k_new=16, k_scale=1.0, v_scale=1.0)
    a.update(kw)
    rc = lib.pa_decode_fp8_append(16, 16, a["k_new"], 16, 16, 16, 16, 16, 1, 8, 8, 128, 16, 4, 0.1, a["k_scale"],
                                  a["v_scale"], 0, 0, None, 0, 0, None)
    assert rc == code


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(k_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(v_new=24), binding.PA_ERR_INVALID_ARG),  # misaligned
        (dict(dtype=binding.PA_F32), binding.PA_ERR_UNSUPPORTED),
        (dict(num_queries=0), binding.PA_ERR_INVALID_ARG),
        (dict(num_queries=5), binding.PA_ERR_UNSUPPORTED),  # group 8 x 5 queries = 40 > 32 columns
    ],
)
def test_decode_mq_append_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(k_new=16, v_new=16, dtype=binding.PA_BF16, num_queries=2)
    a.update(kw)
    rc = lib.pa_decode_mq_append(16, 16, a["k_new"], a["v_new"], 16, 16, 16, 16, 1, a["num_queries"], 32, 4, 128,
                                 16, 4, 0.1, 0, a["dtype"], 0, None, 0, 0, None)
    assert rc == code
    assert lib.pa_last_error().decode()


def test_workspace_size_formula(lib):
    def up(x):
        return (x + 255) // 256 * 256

    S, H, Hk, D, R = 64, 32, 8, 128, 100
    want = up(4 * R * 2 * H * 2) + up(4 * R * 2 * H * D) + up(4 * S * Hk)
    assert lib.pa_decode_workspace_size(S, H, Hk, D, R) == want
    assert lib.pa_decode_workspace_size(0, H, Hk, D, R) == 0
    assert lib.pa_decode_workspace_size(S, 12, 8, D, R) == 0


def test_schedule_partition_host_check(tmp_path):
    """The tile-range decomposition covers every tile once and its partial
    slots never collide (plain C++ build of the shared header)."""
    exe = tmp_path / "schedule_check"
    src = os.path.join(ROOT, "tests", "host", "schedule_check.cpp")
    inc = os.path.join(ROOT, "paged_kv_cache_292_gb300", "csrc")
    subprocess.run(["g++", "-O2", "-std=c++17", "-I" + inc, src, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok")


def test_stall_hook_checks_its_argument(lib):
    """The bounded-wait test hook only records a setting on the host."""
    assert lib.pa_test_stall_copy(-2, 0) == binding.PA_ERR_INVALID_ARG
    assert lib.pa_test_stall_copy(5, 1000) == binding.PA_OK
    assert lib.pa_test_stall_copy(-1, 0) == binding.PA_OK  # cleared


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(k_new=None), binding.PA_ERR_INVALID_ARG),
        (dict(v_new=24), binding.PA_ERR_INVALID_ARG),  # misaligned
        (dict(num_queries=0), binding.PA_ERR_INVALID_ARG),
        (dict(num_queries=5), binding.PA_ERR_UNSUPPORTED),  # group 8 x 5 queries = 40 > 32 columns
        (dict(k_scale=0.0), binding.PA_ERR_INVALID_ARG),
        (dict(v_scale=float("nan")), binding.PA_ERR_INVALID_ARG),
    ],
)
def test_decode_fp8_mq_append_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(k_new=16, v_new=16, num_queries=2, k_scale=1.0, v_scale=1.0)
    a.update(kw)
    rc = lib.pa_decode_fp8_mq_append(16, 16, a["k_new"], a["v_new"], 16, 16, 16, 16, 1, a["num_queries"], 32, 4,
                                     128, 16, 4, 0.1, a["k_scale"], a["v_scale"], 0, 0, None, 0, 0, None)
    assert rc == code
    assert lib.pa_last_error().decode()


@pytest.mark.parametrize(
    "kw, code",
    [
        (dict(query=None), binding.PA_ERR_INVALID_ARG),
        (dict(num_queries=9, heads=16, kv_heads=4), binding.PA_ERR_UNSUPPORTED),  # 4 x 9 = 36 > 32
        (dict(head_size=96), binding.PA_ERR_UNSUPPORTED),
    ],
)
def test_decode_fp8_mq_rejects_bad_arguments_on_host(lib, kw, code):
    a = dict(query=16, num_queries=2, heads=32, kv_heads=8, head_size=128)
    a.update(kw)
    rc = lib.pa_decode_fp8_mq(16, a["query"], 16, 16, 16, 16, 1, a["num_queries"], a["heads"], a["kv_heads"],
                              a["head_size"], 16, 4, 0.1, 1.0, 1.0, 0, 0, None, 0, 0, None)
    assert rc == code
