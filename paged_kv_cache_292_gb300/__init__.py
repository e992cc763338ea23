"""GB300-native paged decode attention (PagedAttention) behind a C ABI.

The compute lives in ``libpagedattn.so`` (hand-written CUDA for sm_103a).  The
Python layer in :mod:`paged_kv_cache_292_gb300.binding` only marshals
arguments into that library; :mod:`paged_kv_cache_292_gb300.workloads` builds
seeded synthetic inputs.
"""

__all__ = ["binding", "workloads"]
