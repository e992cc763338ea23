"""Seeded synthetic decode batches (inputs only; no attention arithmetic).

This module builds the inputs that both the CUDA path and the fp64 oracle are
fed: queries, a paged K/V pool, block tables, context lengths, and one step's
new K/V rows with their slot mapping.  It computes nothing the method computes:
it only draws random numbers and lays values out in the paged pool the way a
block manager would (a sequence's logical block ``j`` lives in physical block
``block_tables[s, j]``).

Every random draw comes from ``numpy.random.default_rng`` (PCG64) seeded with
``[workload_seed, stream_tag, ...]``.  Values are N(0, 1) float32; bf16 inputs
are the round-to-nearest-even cast of those floats (``torch.Tensor.to``).

Per-sequence K/V values are drawn per *logical* token, so the same workload at
block_size 16 and 32 holds the same logical K/V (only the pool layout differs).

The named workloads mirror the decode batches the method is measured on:

=============  =====  ====  =========  ====  ==  ===============================
name           dtype  S     H/Hk       D     bs  context lengths
=============  =====  ====  =========  ====  ==  ===============================
tiny_fp32      f32    4     8/8        64    16  uniform [1, 200], pool 64 blocks
llama3_8b      bf16   64    32/8       128   16  uniform [512, 4096], pool 32768
long_ctx       bf16   8     32/8       128   16  32768 each, pool 18022 (+10%)
mixed_prefix   bf16   256   32/8       128   16  lognormal(median 800, sigma 1),
                                                 clipped [1, 8192]; even seqs
                                                 share a 1024-token prefix
gqa8_70b       bf16   128   64/8       128   16  uniform [1, 16384]; pool = need
                                         or 32   + 10%
=============  =====  ====  =========  ====  ==  ===============================
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

__all__ = ["WorkloadSpec", "Workload", "SPECS", "spec", "make_workload", "kv_bytes_per_token",
           "multi_query_step"]

# Stream tags for the seeded generators.
_CTX, _PERM, _Q, _PREFIX_K, _PREFIX_V, _SEQ_K, _SEQ_V = 1, 2, 3, 4, 5, 10, 11


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    seed: int
    dtype: str  # "f32" or "bf16"
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    ctx_kind: str  # "uniform" | "const" | "lognormal"
    ctx_lo: int
    ctx_hi: int
    ctx_median: float = 0.0
    ctx_sigma: float = 0.0
    pool_blocks: int = 0  # fixed pool size; 0 = need * pool_slack
    pool_slack: float = 1.1
    max_context: int = 0  # max_blocks_per_seq = ceil(max_context / block_size)
    prefix_tokens: int = 0  # shared prefix length for even sequences
    block_assign: str = "shuffle"  # "shuffle" | "contiguous"


SPECS = {
    "tiny_fp32": WorkloadSpec(
        "tiny_fp32", 0, "f32", 4, 8, 8, 64, 16, "uniform", 1, 200, pool_blocks=64, max_context=208
    ),
    "llama3_8b": WorkloadSpec(
        "llama3_8b", 1, "bf16", 64, 32, 8, 128, 16, "uniform", 512, 4096, pool_blocks=32768, max_context=4096
    ),
    "long_ctx": WorkloadSpec(
        "long_ctx", 2, "bf16", 8, 32, 8, 128, 16, "const", 32768, 32768, pool_blocks=18022, max_context=32768
    ),
    "mixed_prefix": WorkloadSpec(
        "mixed_prefix", 3, "bf16", 256, 32, 8, 128, 16, "lognormal", 1, 8192,
        ctx_median=800.0, ctx_sigma=1.0, max_context=8192, prefix_tokens=1024,
    ),
    "gqa8_70b": WorkloadSpec(
        "gqa8_70b", 4, "bf16", 128, 64, 8, 128, 16, "uniform", 1, 16384, max_context=16384
    ),
}


def spec(name: str, **overrides) -> WorkloadSpec:
    """A named spec, optionally with fields replaced (e.g. a smaller batch)."""
    return dataclasses.replace(SPECS[name], **overrides)


def kv_bytes_per_token(s: WorkloadSpec) -> int:
    """K plus V bytes one token occupies across all KV heads."""
    elt = 4 if s.dtype == "f32" else 2
    return 2 * s.num_kv_heads * s.head_size * elt


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    scale: float
    num_blocks: int
    max_blocks_per_seq: int
    q: torch.Tensor  # [S, H, D]
    k_cache: torch.Tensor  # [NB, bs, Hk, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor  # int32 [S, MB]; unused entries -1
    context_lens: torch.Tensor  # int32 [S]
    slot_mapping: torch.Tensor  # int64 [S]: the slot of each sequence's newest token
    k_new: torch.Tensor  # [S, Hk, D]: that token's K (and V below)
    v_new: torch.Tensor
    prewritten: bool  # True: the newest token is already in the pool
    shared_blocks: int  # physical blocks referenced by more than one sequence

    @property
    def torch_dtype(self):
        return torch.float32 if self.spec.dtype == "f32" else torch.bfloat16

    def unique_blocks(self) -> int:
        bt = self.block_tables
        return int(torch.unique(bt[bt >= 0]).numel())


def _draw_context_lens(s: WorkloadSpec) -> np.ndarray:
    rng = np.random.default_rng([s.seed, _CTX])
    if s.ctx_kind == "uniform":
        ctx = rng.integers(s.ctx_lo, s.ctx_hi + 1, s.num_seqs)
    elif s.ctx_kind == "const":
        ctx = np.full(s.num_seqs, s.ctx_lo)
    elif s.ctx_kind == "lognormal":
        draw = np.exp(math.log(s.ctx_median) + s.ctx_sigma * rng.standard_normal(s.num_seqs))
        ctx = np.clip(np.rint(draw), s.ctx_lo, s.ctx_hi)
    else:
        raise ValueError(s.ctx_kind)
    ctx = ctx.astype(np.int64)
    if s.prefix_tokens:
        # Sharing sequences (even index) hold the common prefix plus their own
        # continuation, capped at the maximum context.
        share = np.arange(s.num_seqs) % 2 == 0
        ctx[share] = np.minimum(s.prefix_tokens + ctx[share], s.max_context)
    return ctx


def _normal(rng, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def make_workload(
    spec_or_name,
    *,
    block_size: Optional[int] = None,
    prewritten: bool = True,
    poison: bool = False,
    context_lens: Optional[np.ndarray] = None,
    **overrides,
) -> Workload:
    """Build one seeded decode batch on the CPU.

    block_size   -- override the spec's block size (same logical K/V values).
    prewritten   -- True: every sequence's newest token (position ctx-1) is in
                    the pool already.  False: that slot is left unwritten (zero,
                    or NaN when poisoned) and ``k_new/v_new/slot_mapping`` carry
                    it, to be scattered by the cache-write step.
    poison       -- fill every pool slot that no valid token occupies with NaN.
    context_lens -- explicit per-sequence lengths (overrides the spec's draw).
    """
    s = SPECS[spec_or_name] if isinstance(spec_or_name, str) else spec_or_name
    if overrides:
        s = dataclasses.replace(s, **overrides)
    if block_size is not None:
        s = dataclasses.replace(s, block_size=block_size)
    bs = s.block_size
    S, H, Hk, D = s.num_seqs, s.num_heads, s.num_kv_heads, s.head_size
    tdtype = torch.float32 if s.dtype == "f32" else torch.bfloat16

    ctx = np.asarray(context_lens, dtype=np.int64) if context_lens is not None else _draw_context_lens(s)
    assert ctx.shape == (S,)
    max_ctx = max(s.max_context, int(ctx.max(initial=0)))
    mb = max(1, -(-max_ctx // bs))
    nblk = -(-ctx // bs)

    prefix_blocks = s.prefix_tokens // bs if s.prefix_tokens else 0
    sharing = (np.arange(S) % 2 == 0) if prefix_blocks else np.zeros(S, dtype=bool)
    private_need = int(sum(int(n) - (prefix_blocks if sharing[i] else 0) for i, n in enumerate(nblk)))
    need = private_need + prefix_blocks
    nb = s.pool_blocks if s.pool_blocks else max(1, int(math.ceil(need * s.pool_slack)))
    if need > nb:
        raise ValueError(f"pool of {nb} blocks cannot hold {need}")

    # Physical block assignment: a seeded shuffle of the pool (or identity).
    if s.block_assign == "shuffle":
        order = np.random.default_rng([s.seed, _PERM]).permutation(nb)
    else:
        order = np.arange(nb)
    cursor = 0
    prefix_ids = order[cursor : cursor + prefix_blocks]
    cursor += prefix_blocks
    bt = np.full((S, mb), -1, dtype=np.int32)
    for i in range(S):
        n = int(nblk[i])
        if sharing[i]:
            bt[i, :prefix_blocks] = prefix_ids
            own = n - prefix_blocks
            bt[i, prefix_blocks:n] = order[cursor : cursor + own]
            cursor += own
        else:
            bt[i, :n] = order[cursor : cursor + n]
            cursor += n

    fill = float("nan") if poison else 0.0
    k_cache = torch.full((nb, bs, Hk, D), fill, dtype=tdtype)
    v_cache = torch.full((nb, bs, Hk, D), fill, dtype=tdtype)

    k_new = torch.zeros((S, Hk, D), dtype=tdtype)
    v_new = torch.zeros((S, Hk, D), dtype=tdtype)
    slots = np.full(S, -1, dtype=np.int64)

    prefix_k = prefix_v = None
    if prefix_blocks:
        rk = np.random.default_rng([s.seed, _PREFIX_K])
        rv = np.random.default_rng([s.seed, _PREFIX_V])
        prefix_k = torch.from_numpy(_normal(rk, (s.prefix_tokens, Hk, D))).to(tdtype)
        prefix_v = torch.from_numpy(_normal(rv, (s.prefix_tokens, Hk, D))).to(tdtype)
        _place(k_cache, prefix_ids, prefix_k, bs)
        _place(v_cache, prefix_ids, prefix_v, bs)

    for i in range(S):
        c = int(ctx[i])
        if c == 0:
            continue
        start = s.prefix_tokens if sharing[i] else 0
        rk = np.random.default_rng([s.seed, _SEQ_K, i])
        rv = np.random.default_rng([s.seed, _SEQ_V, i])
        own_k = torch.from_numpy(_normal(rk, (c - start, Hk, D))).to(tdtype)
        own_v = torch.from_numpy(_normal(rv, (c - start, Hk, D))).to(tdtype)
        # Tokens [start, c): the last one is the step's new token.
        k_new[i] = own_k[-1]
        v_new[i] = own_v[-1]
        last = c - 1
        slots[i] = int(bt[i, last // bs]) * bs + last % bs
        keep = c - start if prewritten else c - start - 1
        first_blk = start // bs
        _place(k_cache, bt[i, first_blk : -(-(start + keep) // bs)], own_k[:keep], bs)
        _place(v_cache, bt[i, first_blk : -(-(start + keep) // bs)], own_v[:keep], bs)

    q = torch.from_numpy(_normal(np.random.default_rng([s.seed, _Q]), (S, H, D))).to(tdtype)
    shared = prefix_blocks if int(sharing.sum()) > 1 else 0
    return Workload(
        spec=s,
        scale=1.0 / math.sqrt(D),
        num_blocks=nb,
        max_blocks_per_seq=mb,
        q=q,
        k_cache=k_cache,
        v_cache=v_cache,
        block_tables=torch.from_numpy(bt),
        context_lens=torch.from_numpy(ctx.astype(np.int32)),
        slot_mapping=torch.from_numpy(slots),
        k_new=k_new,
        v_new=v_new,
        prewritten=prewritten,
        shared_blocks=shared,
    )


def _place(pool: torch.Tensor, block_ids, rows: torch.Tensor, bs: int) -> None:
    """Store consecutive logical token rows into the listed physical blocks."""
    n = rows.shape[0]
    if n == 0:
        return
    full = n // bs
    ids = torch.as_tensor(np.asarray(block_ids, dtype=np.int64))
    if full:
        pool[ids[:full]] = rows[: full * bs].reshape(full, bs, *rows.shape[1:])
    rem = n - full * bs
    if rem:
        pool[int(ids[full]), :rem] = rows[full * bs :]


def multi_query_step(w: Workload, num_queries: int):
    """Inputs of a step with ``num_queries`` new tokens per sequence, at
    positions ctx - Q .. ctx - 1 of each sequence: their query rows
    ``q[S, Q, H, D]``, their K/V rows ``k_new, v_new[S * Q, Hk, D]`` (row
    s * Q + i for position ctx - Q + i) and the pool slot of each row
    (``slots[S * Q]``, int64; -1 for a position before the sequence's start).
    Drawn N(0, 1) from one seeded torch generator, q first, then K, then V,
    and cast to the workload's dtype.
    """
    s = w.spec
    S, H, D = w.q.shape
    Q, Hk, bs = num_queries, s.num_kv_heads, s.block_size
    gen = torch.Generator().manual_seed(s.seed + 77)
    q = torch.randn(S, Q, H, D, generator=gen).to(w.q.dtype)
    k_new = torch.randn(S * Q, Hk, D, generator=gen).to(w.q.dtype)
    v_new = torch.randn(S * Q, Hk, D, generator=gen).to(w.q.dtype)
    slots = []
    for i, c in enumerate(w.context_lens.tolist()):
        for j in range(Q):
            pos = c - Q + j
            slots.append(-1 if pos < 0 else int(w.block_tables[i, pos // bs]) * bs + pos % bs)
    return q, k_new, v_new, torch.tensor(slots, dtype=torch.int64)
