"""ctypes binding of libpagedattn.so (argument marshalling only).

The functions named ``pa_*`` mirror the C entry points of ``include/pagedattn.h``
one to one: tensors are passed as their device pointers, sizes as ints, the
stream as the current torch CUDA stream unless one is given.  ``decode`` and
``write_cache`` derive the sizes from tensor shapes and call the same entry
points.  Every computation happens in the CUDA library; if it is missing the
first call raises, there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

from .build import LIB_PATH

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_WORKSPACE = -4
PA_F32 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2
PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_CONTEXT_LEN = 2
PA_DEVERR_SLOT = 4
PA_DEVERR_TIMEOUT = 8

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADER = os.path.join(INCLUDE, "pagedattn.h")
PA_ERR_NO_BLOCKS = -5


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = {
    "pa_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I]),
    "pa_decode_ws": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I, _P, _SZ]),
    "pa_decode_ex": (
        _I,
        [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I, _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_append": (
        _I,
        [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I, _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_fp8_append": (
        _I,
        [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, ctypes.c_float, ctypes.c_float,
         _P, _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "pa_decode_mq": (
        _I,
        [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I, _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_mq_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pa_decode_mq_append": (
        _I,
        [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I, _I, _P, _SZ, _I,
         _P],
    ),
    "pa_write_cache_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, ctypes.c_float, _P, _I, _P]),
    "pa_decode_fp8": (
        _I,
        [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, ctypes.c_float, ctypes.c_float, _P, _I,
         _P, _SZ, _I, _P],
    ),
    "pa_decode_fp8_mq": (
        _I,
        [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, ctypes.c_float, ctypes.c_float, _P,
         _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_fp8_mq_append": (
        _I,
        [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, ctypes.c_float,
         ctypes.c_float, _P, _I, _P, _SZ, _I, _P],
    ),
    "pa_decode_static": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I]),
    "pa_write_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I]),
    "pa_write_cache_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_bm_create": (_P, [_I, _I, _I, _I]),
    "pa_bm_destroy": (None, [_P]),
    "pa_bm_num_free_blocks": (_I, [_P]),
    "pa_bm_context_len": (_I, [_P, _I]),
    "pa_bm_ref_count": (_I, [_P, _I]),
    "pa_bm_append": (_I, [_P, _I, _I, _P, _P, _P]),
    "pa_bm_fork": (_I, [_P, _I, _I]),
    "pa_bm_append_batch": (_I, [_P, _I, _P, _P, _P, _P, _P, _P]),
    "pa_bm_share_prefix": (_I, [_P, _I, _I, _I]),
    "pa_bm_free": (_I, [_P, _I]),
    "pa_bm_export": (_I, [_P, _P, _P]),
    "pa_copy_blocks": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _I]),
    "pa_version": (_I, []),
    "pa_test_stall_copy": (_I, [ctypes.c_longlong, ctypes.c_uint]),
}


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the shared library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def header_symbols() -> list:
    """Names of the functions the public headers (include/*.h) declare."""
    names = set()
    for fn in sorted(os.listdir(INCLUDE)):
        if not fn.endswith(".h"):
            continue
        with open(os.path.join(INCLUDE, fn)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        names |= set(re.findall(r"\b(pa_\w+)\s*\(", text))
    return sorted(names)


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, torch.Tensor):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an int pointer, got {type(x)!r}")


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(rc: int) -> None:
    if rc != PA_OK:
        msg = load().pa_last_error()
        raise PagedAttnError(rc, msg.decode() if msg else "")


def dtype_code(dtype: torch.dtype) -> int:
    if dtype == torch.float32:
        return PA_F32
    if dtype == torch.bfloat16:
        return PA_BF16
    raise ValueError(f"unsupported dtype {dtype}")


# ---- one-to-one entry points -------------------------------------------------


def pa_decode(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
              head_size, block_size, max_blocks_per_seq, scale, stream=None, dtype=None):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            _ptr(context_lens), num_seqs, num_heads, num_kv_heads, head_size, block_size,
                            max_blocks_per_seq, scale, _stream(stream), dtype))


def pa_decode_ws(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                 head_size, block_size, max_blocks_per_seq, scale, stream, dtype, workspace, workspace_bytes):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_ws(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), num_seqs, num_heads, num_kv_heads, head_size, block_size,
                               max_blocks_per_seq, scale, _stream(stream), dtype, _ptr(workspace),
                               workspace_bytes))


def pa_decode_ex(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                 head_size, block_size, max_blocks_per_seq, scale, stream=None, dtype=None,
                 num_physical_blocks=0, workspace=None, workspace_bytes=0, num_ranges=0, error_flag=None):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_ex(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), num_seqs, num_heads, num_kv_heads, head_size, block_size,
                               max_blocks_per_seq, scale, _stream(stream), dtype, num_physical_blocks,
                               _ptr(workspace), workspace_bytes, num_ranges, _ptr(error_flag)))


def pa_decode_static(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads, num_kv_heads,
                     head_size, block_size, max_blocks_per_seq, scale, stream=None, dtype=None):
    """pa_decode without any allocation: scratch is an array compiled into the library."""
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_static(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                   max_blocks_per_seq, scale, _stream(stream), dtype))


def pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, num_ranges=0) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_size, num_ranges))


def pa_decode_mq(out, query, k_cache, v_cache, block_tables, context_lens, num_seqs, num_queries, num_heads,
                 num_kv_heads, head_size, block_size, max_blocks_per_seq, scale, stream=None, dtype=None,
                 num_physical_blocks=0, workspace=None, workspace_bytes=0, num_ranges=0, error_flag=None):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_mq(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                               _ptr(context_lens), num_seqs, num_queries, num_heads, num_kv_heads, head_size,
                               block_size, max_blocks_per_seq, scale, _stream(stream), dtype, num_physical_blocks,
                               _ptr(workspace), workspace_bytes, num_ranges, _ptr(error_flag)))


def pa_decode_mq_workspace_size(num_seqs, num_queries, num_heads, num_kv_heads, head_size, num_ranges=0) -> int:
    return int(load().pa_decode_mq_workspace_size(num_seqs, num_queries, num_heads, num_kv_heads, head_size,
                                                  num_ranges))


def decode_multi(query, k_cache, v_cache, block_tables, context_lens, scale, out=None, stream=None, *,
                 num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """out[S, Q, H, D]: several causal query tokens per sequence (shapes as in ``pa_decode_mq``)."""
    _require_cuda(query, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, Q, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    pa_decode_mq(out, query, k_cache, v_cache, block_tables, context_lens, S, Q, H, Hk, D, bs,
                 block_tables.shape[1], float(scale), stream, dtype_code(query.dtype),
                 NB if check_block_ids else 0, workspace, ws_bytes, num_ranges, error_flag)
    return out


def pa_write_cache(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_size,
                   block_size, num_physical_blocks, stream=None, dtype=None):
    dtype = dtype_code(k_new.dtype) if dtype is None else dtype
    _check(load().pa_write_cache(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                 num_tokens, num_kv_heads, head_size, block_size, num_physical_blocks,
                                 _stream(stream), dtype))


def pa_write_cache_ex(k_new, v_new, slot_mapping, k_cache, v_cache, num_tokens, num_kv_heads, head_size,
                      block_size, num_physical_blocks, stream=None, dtype=None, error_flag=None):
    dtype = dtype_code(k_new.dtype) if dtype is None else dtype
    _check(load().pa_write_cache_ex(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                                    num_tokens, num_kv_heads, head_size, block_size, num_physical_blocks,
                                    _stream(stream), dtype, _ptr(error_flag)))


def pa_last_error() -> str:
    msg = load().pa_last_error()
    return msg.decode() if msg else ""


def pa_version() -> int:
    return int(load().pa_version())


def pa_test_stall_copy(tile: int, wait_limit_us: int = 0) -> None:
    """Test hook: the next decode launch on this thread withholds tile `tile`'s copies and bounds its waits."""
    _check(load().pa_test_stall_copy(tile, wait_limit_us))


# ---- shape-derived conveniences ---------------------------------------------


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def pa_decode_append(out, query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale, stream=None,
                     dtype=None, num_physical_blocks=0, workspace=None, workspace_bytes=0, num_ranges=0,
                     error_flag=None):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_append(_ptr(out), _ptr(query), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), num_seqs, num_heads,
                                   num_kv_heads, head_size, block_size, max_blocks_per_seq, float(scale),
                                   _stream(stream), dtype, num_physical_blocks, _ptr(workspace),
                                   workspace_bytes, num_ranges, _ptr(error_flag)))


def decode_append(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                  stream=None, *, num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """One decode step with the newest token's K/V (k_new/v_new[S, Hk, D]) written into the pools at
    position context_lens[s]-1 by the decode itself (shapes as in ``pa_decode_append``)."""
    _require_cuda(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    pa_decode_append(out, query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, S, H, Hk, D, bs,
                     block_tables.shape[1], float(scale), stream, dtype_code(query.dtype),
                     NB if check_block_ids else 0, workspace, ws_bytes, num_ranges, error_flag)
    return out


def pa_decode_mq_append(out, query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, num_seqs,
                        num_queries, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, scale,
                        stream=None, dtype=None, num_physical_blocks=0, workspace=None, workspace_bytes=0,
                        num_ranges=0, error_flag=None):
    dtype = dtype_code(query.dtype) if dtype is None else dtype
    _check(load().pa_decode_mq_append(_ptr(out), _ptr(query), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), num_seqs, num_queries,
                                      num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
                                      float(scale), _stream(stream), dtype, num_physical_blocks, _ptr(workspace),
                                      workspace_bytes, num_ranges, _ptr(error_flag)))


def decode_multi_append(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, out=None,
                        stream=None, *, num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """Several causal query tokens per sequence with their K/V (k_new/v_new[S*Q, Hk, D], token i of
    sequence s at row s*Q+i, position context_lens[s]-Q+i) written into the pools by the same launch
    (shapes as in ``pa_decode_mq_append``)."""
    _require_cuda(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, Q, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    pa_decode_mq_append(out, query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, S, Q, H, Hk, D,
                        bs, block_tables.shape[1], float(scale), stream, dtype_code(query.dtype),
                        NB if check_block_ids else 0, workspace, ws_bytes, num_ranges, error_flag)
    return out


def decode_fp8_append(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                      v_scale, out=None, stream=None, *, num_ranges=0, workspace=None, error_flag=None,
                      check_block_ids=False):
    """pa_decode_fp8_append: the FP8-pool step with the newest token's quantising write fused in."""
    _require_cuda(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_decode_fp8_append(_ptr(out), _ptr(query), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), S, H, Hk, D, bs,
                                       block_tables.shape[1], float(scale), float(k_scale), float(v_scale),
                                       _stream(stream), NB if check_block_ids else 0, _ptr(workspace), ws_bytes,
                                       num_ranges, _ptr(error_flag)))
    return out


def decode(query, k_cache, v_cache, block_tables, context_lens, scale, out=None, stream=None, *,
           num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """out[S, H, D] = paged decode attention (shapes as in ``pa_decode``)."""
    _require_cuda(query, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    pa_decode_ex(out, query, k_cache, v_cache, block_tables, context_lens, S, H, Hk, D, bs,
                 block_tables.shape[1], float(scale), stream, dtype_code(query.dtype),
                 NB if check_block_ids else 0, workspace, ws_bytes, num_ranges, error_flag)
    return out


def write_cache(k_new, v_new, slot_mapping, k_cache, v_cache, stream=None, *, error_flag=None):
    """Scatter k_new/v_new[T, Hk, D] into the pools at slot_mapping[T] (int64)."""
    _require_cuda(k_new, v_new, slot_mapping, k_cache, v_cache, error_flag)
    T, Hk, D = k_new.shape
    NB, bs = k_cache.shape[:2]
    pa_write_cache_ex(k_new, v_new, slot_mapping, k_cache, v_cache, T, Hk, D, bs, NB, stream,
                      dtype_code(k_new.dtype), error_flag)


def pa_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_kv_heads, head_size, block_size, num_physical_blocks,
                   stream=None, dtype=None):
    dtype = dtype_code(k_cache.dtype) if dtype is None else dtype
    _check(load().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), num_pairs, num_kv_heads, head_size,
                                 block_size, num_physical_blocks, _stream(stream), dtype))


class BlockManager:
    """The C block manager (pa_bm_*): host memory only, no device calls."""

    def __init__(self, num_blocks, block_size, max_seqs, max_blocks_per_seq):
        lib = load()
        self._h = lib.pa_bm_create(num_blocks, block_size, max_seqs, max_blocks_per_seq)
        if not self._h:
            raise PagedAttnError(PA_ERR_INVALID_ARG, pa_last_error())
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_seqs, self.max_blocks_per_seq = max_seqs, max_blocks_per_seq

    def close(self):
        if self._h:
            load().pa_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def num_free_blocks(self):
        return load().pa_bm_num_free_blocks(self._h)

    def context_len(self, seq):
        return load().pa_bm_context_len(self._h, seq)

    def ref_count(self, block):
        return load().pa_bm_ref_count(self._h, block)

    def append(self, seq, num_tokens):
        """Slots (int64 tensor) for num_tokens new tokens, and the list of (src, dst) block copies."""
        slots = torch.empty(max(num_tokens, 1), dtype=torch.int64)
        copies = (ctypes.c_int32 * 2)()
        n = ctypes.c_int(0)
        _check(load().pa_bm_append(self._h, seq, num_tokens, slots.data_ptr(), ctypes.addressof(copies),
                                   ctypes.addressof(n)))
        return slots[:num_tokens], [(copies[0], copies[1])] if n.value else []

    def append_batch(self, seqs, counts, slots_out=None, copies_out=None):
        """One call for many sequences; returns (slots, list of (src, dst) copies)."""
        seqs = torch.as_tensor(seqs, dtype=torch.int32)
        counts = torch.as_tensor(counts, dtype=torch.int32)
        total = int(counts.sum())
        if slots_out is None:
            slots_out = torch.empty(max(total, 1), dtype=torch.int64)
        if copies_out is None:
            copies_out = torch.empty(2 * max(len(seqs), 1), dtype=torch.int32)
        nc, nd = ctypes.c_int(0), ctypes.c_int(0)
        _check(load().pa_bm_append_batch(self._h, len(seqs), seqs.data_ptr(), counts.data_ptr(), slots_out.data_ptr(),
                                         copies_out.data_ptr(), ctypes.addressof(nc), ctypes.addressof(nd)))
        pairs = copies_out[: 2 * nc.value].view(-1, 2)
        return slots_out[:total], [tuple(p) for p in pairs.tolist()]

    def fork(self, parent, child):
        _check(load().pa_bm_fork(self._h, parent, child))

    def share_prefix(self, seq, donor, num_tokens):
        _check(load().pa_bm_share_prefix(self._h, seq, donor, num_tokens))

    def free(self, seq):
        _check(load().pa_bm_free(self._h, seq))

    def export(self):
        tables = torch.empty((self.max_seqs, self.max_blocks_per_seq), dtype=torch.int32)
        lens = torch.empty(self.max_seqs, dtype=torch.int32)
        _check(load().pa_bm_export(self._h, tables.data_ptr(), lens.data_ptr()))
        return tables, lens


def write_cache_fp8(k_new, v_new, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None, *,
                    error_flag=None):
    """Quantise and scatter k_new/v_new[T, Hk, D] (bf16 or f32) into uint8 E4M3 pools."""
    _require_cuda(k_new, v_new, slot_mapping, k_cache, v_cache, error_flag)
    T, Hk, D = k_new.shape
    NB, bs = k_cache.shape[:2]
    _check(load().pa_write_cache_fp8(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), T,
                                     Hk, D, bs, NB, float(k_scale), float(v_scale), _stream(stream),
                                     dtype_code(k_new.dtype), _ptr(error_flag)))


def decode_fp8(query, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale, out=None, stream=None,
               *, num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """out[S, H, D] (bf16) over uint8 E4M3 pools."""
    _require_cuda(query, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_decode_fp8(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                _ptr(context_lens), S, H, Hk, D, bs, block_tables.shape[1], float(scale),
                                float(k_scale), float(v_scale), _stream(stream), NB if check_block_ids else 0,
                                _ptr(workspace), ws_bytes, num_ranges, _ptr(error_flag)))
    return out


def decode_fp8_multi(query, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale, out=None,
                     stream=None, *, num_ranges=0, workspace=None, error_flag=None, check_block_ids=False):
    """out[S, Q, H, D] (bf16): several causal query tokens per sequence over uint8 E4M3 pools."""
    _require_cuda(query, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, Q, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_decode_fp8_mq(_ptr(out), _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                   _ptr(context_lens), S, Q, H, Hk, D, bs, block_tables.shape[1], float(scale),
                                   float(k_scale), float(v_scale), _stream(stream), NB if check_block_ids else 0,
                                   _ptr(workspace), ws_bytes, num_ranges, _ptr(error_flag)))
    return out


def decode_fp8_multi_append(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                            v_scale, out=None, stream=None, *, num_ranges=0, workspace=None, error_flag=None,
                            check_block_ids=False):
    """pa_decode_fp8_mq_append: the FP8 multi-query step with the Q new rows' quantising write fused in."""
    _require_cuda(query, k_new, v_new, k_cache, v_cache, block_tables, context_lens, out, workspace, error_flag)
    S, Q, H, D = query.shape
    NB, bs, Hk, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(query)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().pa_decode_fp8_mq_append(_ptr(out), _ptr(query), _ptr(k_new), _ptr(v_new), _ptr(k_cache),
                                          _ptr(v_cache), _ptr(block_tables), _ptr(context_lens), S, Q, H, Hk, D, bs,
                                          block_tables.shape[1], float(scale), float(k_scale), float(v_scale),
                                          _stream(stream), NB if check_block_ids else 0, _ptr(workspace), ws_bytes,
                                          num_ranges, _ptr(error_flag)))
    return out
