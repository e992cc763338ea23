"""FP8 E4M3 codec and the quantised-cache reference (test infrastructure only).

The pages name quantisation as a vLLM feature but give no format.  The reading
taken: the KV pool stores E4M3 values (1 sign bit, 4 exponent bits with bias
7, 3 mantissa bits; no infinities; the all-ones exponent and mantissa is NaN;
largest finite magnitude 448) with one float scale per pool: a stored code c
stands for decode(c) * scale.  Encoding divides by the scale and rounds to the
nearest representable value, ties to even, saturating at +-448.

This module writes the format out from that definition (bit fields, not a
library call) so the CUDA path's conversions can be checked against it.
"""

from __future__ import annotations

import numpy as np

import oracle.paged_attention as pa

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of each E4M3 code (uint8)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = sign * (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    subnormal = sign * (man / 8.0) * 2.0**-6
    out = np.where(exp == 0, subnormal, normal)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, out)


def _all_finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = e4m3_decode(codes)
    keep = np.isfinite(vals)
    return codes[keep], vals[keep]


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code to each value (ties to the even code), saturating.

    Brute force over the 127 non-negative finite codes: pick the closest
    magnitude; on a tie the candidate with an even mantissa (lowest bit 0)
    wins.  The sign bit is the input's (so a negative value that rounds to
    zero gives the negative zero 0x80, as IEEE rounding does).
    """
    x = np.asarray(x, dtype=np.float64)
    codes, vals = _all_finite_codes()
    pos = codes < 0x80
    pcodes, pvals = codes[pos], vals[pos]  # 0 .. 448, 127 codes
    order = np.argsort(pvals)
    pcodes, pvals = pcodes[order], pvals[order]
    a = np.minimum(np.abs(x), E4M3_MAX)
    idx = np.searchsorted(pvals, a)  # first value >= a
    hi = np.clip(idx, 0, len(pvals) - 1)
    lo = np.clip(idx - 1, 0, len(pvals) - 1)
    d_hi = pvals[hi] - a
    d_lo = a - pvals[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & ((pcodes[lo] & 1) == 0))
    mag = np.where(take_lo, pcodes[lo], pcodes[hi]).astype(np.uint8)
    return np.where(np.signbit(x), mag | 0x80, mag).astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """Code of x / scale.  The quotient is taken in float32 (IEEE division, as
    the CUDA write does) and then rounded to E4M3: both sides decide each code
    in the same precision."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return e4m3_encode(q.astype(np.float64))


def write_cache_fp8(k_cache, v_cache, k_new, v_new, slot_mapping, block_size, k_scale, v_scale):
    """Quantised cache write: the scatter of paged_attention.write_cache applied
    to quantize(k_new, k_scale) and quantize(v_new, v_scale)."""
    return pa.write_cache(k_cache, v_cache, quantize(k_new, k_scale), quantize(v_new, v_scale),
                          slot_mapping, block_size)


def decode_fp8(q, k_codes, v_codes, block_tables, context_lens, scale, block_size, k_scale, v_scale):
    """Paged decode over the dequantised pools (decode(c) * scale), fp64."""
    kc = e4m3_decode(k_codes) * k_scale
    vc = e4m3_decode(v_codes) * v_scale
    return pa.decode(q, kc, vc, block_tables, context_lens, scale, block_size)
