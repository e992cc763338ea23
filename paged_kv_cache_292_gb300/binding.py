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
PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_CONTEXT_LEN = 2
PA_DEVERR_SLOT = 4
PA_DEVERR_TIMEOUT = 8

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pagedattn.h")


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
    "pa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "pa_decode_static": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _I]),
    "pa_write_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I]),
    "pa_write_cache_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _P]),
    "pa_last_error": (ctypes.c_char_p, []),
    "pa_version": (_I, []),
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
    """Names of the functions the public header declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_\w+)\s*\(", text)))


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


# ---- shape-derived conveniences ---------------------------------------------


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


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
