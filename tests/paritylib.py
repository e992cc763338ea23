"""Helpers shared by the GPU parity tests: move a seeded workload to the
device, run the fp64 oracle on (a sample of) its sequences, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": (1e-5, None), "bf16": (1e-2, 1e-3)}  # (max-abs, mean-abs)


def int_view(dtype: str):
    return torch.int32 if dtype == "f32" else torch.int16


def to_device(w, dev="cuda"):
    return {
        k: getattr(w, k).to(dev)
        for k in ("q", "k_cache", "v_cache", "block_tables", "context_lens", "slot_mapping", "k_new", "v_new")
    }


def oracle_pools_after_write(w):
    """fp64 pools after the oracle's cache write (inputs from the generator)."""
    view = int_view(w.spec.dtype)
    k2, v2 = oracle.write_cache(
        w.k_cache.view(view).numpy(), w.v_cache.view(view).numpy(), w.k_new.view(view).numpy(),
        w.v_new.view(view).numpy(), w.slot_mapping.numpy(), w.spec.block_size,
    )
    return torch.from_numpy(k2).view(w.k_cache.dtype), torch.from_numpy(v2).view(w.v_cache.dtype)


def oracle_decode(w, k_cache=None, v_cache=None, seqs=None):
    """Oracle output for the listed sequences (all by default), in float64.

    Only the physical blocks those sequences use are widened to fp64: the pool
    is compacted and the tables relabelled (a relabelling the oracle is pinned
    to be invariant under).
    """
    k_cache = w.k_cache if k_cache is None else k_cache
    v_cache = w.v_cache if v_cache is None else v_cache
    bs = w.spec.block_size
    seqs = list(range(w.spec.num_seqs)) if seqs is None else list(seqs)
    ctx = w.context_lens.numpy()[seqs]
    bt = w.block_tables.numpy()[seqs]
    nblk = [-(-int(c) // bs) for c in ctx]
    used = sorted({int(b) for i, n in enumerate(nblk) for b in bt[i, :n]})
    remap = {b: i for i, b in enumerate(used)}
    bt2 = np.full((len(seqs), max(1, max(nblk, default=1))), -1, dtype=np.int64)
    for i, n in enumerate(nblk):
        bt2[i, :n] = [remap[int(b)] for b in bt[i, :n]]
    idx = torch.as_tensor(used if used else [0], dtype=torch.long)
    kc = k_cache[idx].double().numpy()
    vc = v_cache[idx].double().numpy()
    q = w.q[seqs].double().numpy()
    return oracle.decode(q, kc, vc, bt2, ctx, w.scale, bs)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0**-126)))
    return 2.0 ** (e - 8)


def assert_close(got: torch.Tensor, want: np.ndarray, dtype: str, what: str = ""):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - want)
    max_tol, mean_tol = TOL[dtype]
    if dtype == "bf16":
        # The result is stored in bf16: rounding it costs up to half an ulp.
        # Below |out| = 4 that is at most 2^-7 and fits inside 1e-2; above it
        # the half ulp alone passes 1e-2, so only the excess over 2^-7 is
        # allowed on top there.  Below 4 the bound stays exactly 1e-2.
        err = np.maximum(err - np.maximum(bf16_half_ulp(want) - 2.0**-7, 0.0), 0.0)
    assert err.max() <= max_tol, f"{what}: max abs err {err.max():.3e} > {max_tol}"
    if mean_tol is not None:
        assert err.mean() <= mean_tol, f"{what}: mean abs err {err.mean():.3e} > {mean_tol}"
    return float(err.max()), float(err.mean())
