"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

The oracle restates the paged gather and "standard attention" of the
PagedAttention kernel description ("vLLM three-process architecture and the
PagedAttention kernel", section 3.2 steps 1-5).  None of these checks re-types
the oracle's own formula: each compares it against an independent fact
(a layout identity, a closed form, a brute-force scalar loop, a library
routine on the textbook special case, or a page's worked allocation).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_292_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def _np(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def _random_paged(rng, S=3, H=4, Hk=2, D=8, bs=4, max_ctx=23, nb=40, ctx=None):
    ctx = rng.integers(1, max_ctx + 1, S) if ctx is None else np.asarray(ctx)
    mb = -(-max_ctx // bs)
    perm = rng.permutation(nb)
    bt = np.full((S, mb), -1, dtype=np.int64)
    cur = 0
    for s in range(S):
        n = -(-int(ctx[s]) // bs)
        bt[s, :n] = perm[cur : cur + n]
        cur += n
    kc = rng.standard_normal((nb, bs, Hk, D))
    vc = rng.standard_normal((nb, bs, Hk, D))
    q = rng.standard_normal((S, H, D))
    return q, kc, vc, bt, ctx


# --- gather ---------------------------------------------------------------


def test_permutation_invariance():
    """(i) Relabelling physical blocks (pool and tables together) changes nothing."""
    rng = np.random.default_rng(1)
    q, kc, vc, bt, ctx = _random_paged(rng)
    out = oracle.decode(q, kc, vc, bt, ctx, 0.35, 4)
    pi = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    bt2 = np.where(bt >= 0, pi[np.clip(bt, 0, None)], -1)
    out2 = oracle.decode(q, kc2, vc2, bt2, ctx, 0.35, 4)
    assert np.array_equal(out, out2)


def test_paged_equals_contiguous():
    """(ii) Paged result == attention over the same K/V stored contiguously.

    The contiguous side uses torch's scaled_dot_product_attention on K/V laid
    out [ctx, D] per head directly, so no block table is involved at all.
    """
    rng = np.random.default_rng(2)
    S, H, Hk, D, bs = 3, 6, 3, 8, 4
    ctx = np.array([1, 9, 17])
    k_logical = [rng.standard_normal((c, Hk, D)) for c in ctx]
    v_logical = [rng.standard_normal((c, Hk, D)) for c in ctx]
    nb = 20
    perm = rng.permutation(nb)
    bt = np.full((S, 5), -1)
    kc = np.full((nb, bs, Hk, D), np.nan)
    vc = np.full((nb, bs, Hk, D), np.nan)
    cur = 0
    for s in range(S):
        for t in range(ctx[s]):
            if t % bs == 0:
                bt[s, t // bs] = perm[cur]
                cur += 1
            kc[bt[s, t // bs], t % bs] = k_logical[s][t]
            vc[bt[s, t // bs], t % bs] = v_logical[s][t]
    q = rng.standard_normal((S, H, D))
    scale = 1 / math.sqrt(D)
    out = oracle.decode(q, kc, vc, bt, ctx, scale, bs)
    G = H // Hk
    for s in range(S):
        qs = torch.from_numpy(q[s])[:, None, :]  # [H, 1, D]
        ks = torch.from_numpy(k_logical[s]).permute(1, 0, 2).repeat_interleave(G, 0)  # [H, ctx, D]
        vs = torch.from_numpy(v_logical[s]).permute(1, 0, 2).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, scale=scale)[:, 0, :]
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=0, atol=1e-13)


def test_block_size_invariance():
    """(iii) The same logical K/V in bs=16 and bs=32 pools give the same output."""
    sp = workloads.spec("gqa8_70b", num_seqs=3, ctx_lo=1, ctx_hi=90, max_context=96)
    w16 = workloads.make_workload(sp, block_size=16)
    w32 = workloads.make_workload(sp, block_size=32)
    args = lambda w: (  # noqa: E731
        _np(w.q), _np(w.k_cache), _np(w.v_cache), w.block_tables.numpy(), w.context_lens.numpy(), w.scale,
    )
    o16 = oracle.decode(*args(w16), 16)
    o32 = oracle.decode(*args(w32), 32)
    assert np.array_equal(o16, o32)


def test_page_toy_allocation_golden():
    """(iv) The preface's toy allocation (A -> B1/B3/B7, B -> B2/B5), closed form."""
    with open(os.path.join(HERE, "golden", "p2_toy_allocation.json")) as f:
        g = json.load(f)
    bs, nb, H, Hk, D = g["block_size"], g["num_blocks"], g["num_heads"], g["num_kv_heads"], g["head_size"]
    bt = np.array(g["block_tables"])
    ctx = np.array(g["context_lens"])
    kc = np.full((nb, bs, Hk, D), np.nan)
    vc = np.full((nb, bs, Hk, D), np.nan)
    for s in range(len(ctx)):
        for t in range(ctx[s]):
            kc[bt[s, t // bs], t % bs, 0] = [1.0, 1.0]
            vc[bt[s, t // bs], t % bs, 0] = [t, 100 * s + 2 * t]
    q = np.array(g["query"])
    out = oracle.decode(q, kc, vc, bt, ctx, 1 / math.sqrt(D), bs)
    np.testing.assert_allclose(out, np.array(g["expected_out"]), rtol=0, atol=1e-12)
    # Free blocks (B4, B6, ...) hold NaN and must never be read.
    assert np.all(np.isfinite(out))


# --- attention ------------------------------------------------------------


def test_context_one_returns_v():
    """(v) With one valid token every weight is 1: out == v_0 exactly."""
    rng = np.random.default_rng(3)
    q, kc, vc, bt, _ = _random_paged(rng, ctx=[1, 1, 1])
    out = oracle.decode(q, kc, vc, bt, [1, 1, 1], 0.7, 4)
    G = q.shape[1] // kc.shape[2]
    for s in range(3):
        for h in range(q.shape[1]):
            assert np.array_equal(out[s, h], vc[bt[s, 0], 0, h // G])


def test_identical_keys_and_zero_scale_give_mean_of_v():
    """(vi) Equal scores -> uniform weights -> mean of the gathered V rows."""
    rng = np.random.default_rng(4)
    q, kc, vc, bt, ctx = _random_paged(rng)
    kc_same = np.broadcast_to(rng.standard_normal((1, 1, kc.shape[2], kc.shape[3])), kc.shape).copy()
    G = q.shape[1] // kc.shape[2]
    for kcache, scale in ((kc_same, 0.5), (kc, 0.0)):
        out = oracle.decode(q, kcache, vc, bt, ctx, scale, 4)
        for s in range(q.shape[0]):
            rows = np.stack([vc[bt[s, t // 4], t % 4] for t in range(ctx[s])])  # [ctx, Hk, D]
            for h in range(q.shape[1]):
                np.testing.assert_allclose(out[s, h], rows[:, h // G].mean(axis=0), rtol=0, atol=1e-13)


def test_weights_sum_to_one_and_are_positive():
    """(vii) Softmax weights are a probability vector per head."""
    rng = np.random.default_rng(5)
    q_s = rng.standard_normal((8, 16)) * 3
    k_s = rng.standard_normal((37, 2, 16)) * 3
    p = oracle.attention_weights(q_s, k_s, 0.25)
    assert np.all(p > 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)


def test_key_shift_invariance():
    """(viii) k_t -> k_t + c shifts every score of a head by the same q.c."""
    rng = np.random.default_rng(6)
    q, kc, vc, bt, ctx = _random_paged(rng)
    c = rng.standard_normal(kc.shape[3])
    out = oracle.decode(q, kc, vc, bt, ctx, 0.3, 4)
    out2 = oracle.decode(q, kc + c, vc, bt, ctx, 0.3, 4)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)


def test_affine_in_v():
    """(ix) V + c -> out + c; a constant V gives that constant."""
    rng = np.random.default_rng(7)
    q, kc, vc, bt, ctx = _random_paged(rng)
    c = rng.standard_normal(vc.shape[3])
    out = oracle.decode(q, kc, vc, bt, ctx, 0.3, 4)
    out2 = oracle.decode(q, kc, vc + c, bt, ctx, 0.3, 4)
    np.testing.assert_allclose(out2, out + c, rtol=0, atol=1e-12)
    const = oracle.decode(q, kc, np.full_like(vc, 2.5), bt, ctx, 0.3, 4)
    np.testing.assert_allclose(const, 2.5, rtol=0, atol=1e-13)


def test_one_dominant_key():
    """(x) A score gap of g leaves the other tokens a total weight below (n-1)e^{-g}."""
    rng = np.random.default_rng(8)
    D, n = 16, 30
    k_s = rng.standard_normal((n, 1, D))
    v_s = rng.standard_normal((n, 1, D))
    j = 17
    q_s = (k_s[j, 0] * 50.0)[None, :]
    x = k_s[:, 0, :] @ q_s[0]
    gap = x[j] - np.max(np.delete(x, j))
    assert gap > 30  # scores in the thousands: a missing max-subtraction overflows
    out = oracle.attention(q_s, k_s, v_s, 1.0)
    bound = (n - 1) * math.exp(-gap) * 2 * np.abs(v_s).max()
    np.testing.assert_allclose(out[0], v_s[j, 0], rtol=0, atol=max(bound, 1e-15))
    assert np.all(np.isfinite(out))


def _brute_force(q, kc, vc, bt, ctx, scale, bs):
    """Scalar loops with math.exp: a second, independent statement of the op."""
    S, H, D = q.shape
    Hk = kc.shape[2]
    G = H // Hk
    out = [[[0.0] * D for _ in range(H)] for _ in range(S)]
    for s in range(S):
        for h in range(H):
            kv = h // G
            scores = []
            for t in range(int(ctx[s])):
                blk, off = int(bt[s][t // bs]), t % bs
                dot = 0.0
                for d in range(D):
                    dot += float(q[s][h][d]) * float(kc[blk][off][kv][d])
                scores.append(scale * dot)
            if not scores:
                continue
            mx = max(scores)
            w = [math.exp(x - mx) for x in scores]
            tot = sum(w)
            for d in range(D):
                acc = 0.0
                for t in range(int(ctx[s])):
                    blk, off = int(bt[s][t // bs]), t % bs
                    acc += w[t] * float(vc[blk][off][kv][d])
                out[s][h][d] = acc / tot
    return np.array(out)


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_tiny(seed):
    """(xi) Tiny random cases (S<=2, ctx<=5, D<=4, GQA) against scalar loops."""
    rng = np.random.default_rng(100 + seed)
    Hk = int(rng.integers(1, 3))
    H = Hk * int(rng.integers(1, 4))
    D = int(rng.integers(1, 5))
    S = int(rng.integers(1, 3))
    q, kc, vc, bt, ctx = _random_paged(rng, S=S, H=H, Hk=Hk, D=D, bs=2, max_ctx=5, nb=8)
    scale = float(rng.uniform(0.1, 2.0))
    np.testing.assert_allclose(
        oracle.decode(q, kc, vc, bt, ctx, scale, 2), _brute_force(q, kc, vc, bt, ctx, scale, 2), rtol=0, atol=1e-13
    )


def test_gqa_matches_sdpa_with_repeated_kv_heads():
    """(xii) GQA decode == torch SDPA (CPU, fp64) with each KV head repeated G times."""
    rng = np.random.default_rng(9)
    S, H, Hk, D, bs = 2, 8, 2, 16, 8
    q, kc, vc, bt, ctx = _random_paged(rng, S=S, H=H, Hk=Hk, D=D, bs=bs, max_ctx=40, nb=16)
    out = oracle.decode(q, kc, vc, bt, ctx, 0.2, bs)
    for s in range(S):
        flat_k = kc.reshape(-1, Hk, D)
        flat_v = vc.reshape(-1, Hk, D)
        idx = [bt[s, t // bs] * bs + t % bs for t in range(ctx[s])]
        ks = torch.from_numpy(flat_k[idx]).permute(1, 0, 2).repeat_interleave(H // Hk, 0)
        vs = torch.from_numpy(flat_v[idx]).permute(1, 0, 2).repeat_interleave(H // Hk, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(torch.from_numpy(q[s])[:, None], ks, vs, scale=0.2)
        np.testing.assert_allclose(out[s], ref[:, 0].numpy(), rtol=0, atol=1e-13)


def test_empty_context_is_zero():
    rng = np.random.default_rng(10)
    q, kc, vc, bt, _ = _random_paged(rng, ctx=[0, 3, 0])
    out = oracle.decode(q, kc, vc, bt, [0, 3, 0], 0.5, 4)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out))


# --- split + merge --------------------------------------------------------


@pytest.mark.parametrize("part", [1, 3, 4, 16, 64])
def test_split_merge_equals_unsplit(part):
    """(xiii) Any partition size, merged by log-sum-exp, equals the unsplit softmax."""
    rng = np.random.default_rng(11)
    q, kc, vc, bt, ctx = _random_paged(rng, S=3, max_ctx=41, nb=40, ctx=[41, 1, 17])
    ref = oracle.decode(q, kc, vc, bt, ctx, 0.4, 4)
    out = oracle.decode_split(q, kc, vc, bt, ctx, 0.4, 4, part)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-13)


def test_merge_of_single_partition_is_identity():
    m = np.array([[0.5, -1.0]])
    l = np.array([[2.0, 4.0]])
    o = np.array([[[2.0, 4.0], [8.0, -4.0]]])
    np.testing.assert_allclose(oracle.merge_partials(m, l, o), [[1.0, 2.0], [2.0, -1.0]])


# --- write cache ----------------------------------------------------------


def test_write_cache_bit_exact_and_local():
    """(xiv) The scatter writes exactly the addressed rows, bit for bit."""
    rng = np.random.default_rng(12)
    nb, bs, Hk, D, T = 6, 4, 2, 8, 5
    kc = rng.integers(-(2**15), 2**15, (nb, bs, Hk, D)).astype(np.int16)
    vc = rng.integers(-(2**15), 2**15, (nb, bs, Hk, D)).astype(np.int16)
    kn = rng.integers(-(2**15), 2**15, (T, Hk, D)).astype(np.int16)
    vn = rng.integers(-(2**15), 2**15, (T, Hk, D)).astype(np.int16)
    slots = np.array([0, 23, -1, 9, 14])
    k2, v2 = oracle.write_cache(kc, vc, kn, vn, slots, bs)
    touched = set()
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        touched.add((sl // bs, sl % bs))
        assert np.array_equal(k2[sl // bs, sl % bs], kn[i])
        assert np.array_equal(v2[sl // bs, sl % bs], vn[i])
    for b in range(nb):
        for o in range(bs):
            if (b, o) not in touched:
                assert np.array_equal(k2[b, o], kc[b, o]) and np.array_equal(v2[b, o], vc[b, o])
    # inputs untouched
    assert not np.shares_memory(k2, kc)


@pytest.mark.parametrize("name", ["tiny_fp32", "mixed_small"])
def test_write_then_decode_equals_prewritten_pool(name):
    """(xiv) Writing each sequence's newest token then decoding equals decoding
    the pool the generator laid out with that token already in place."""
    if name == "mixed_small":
        sp = workloads.spec("mixed_prefix", num_seqs=6, ctx_median=20.0, ctx_hi=64, max_context=96, prefix_tokens=32)
    else:
        sp = workloads.spec(name)
    pre = workloads.make_workload(sp, prewritten=True, poison=True)
    post = workloads.make_workload(sp, prewritten=False, poison=True)
    view = torch.int32 if sp.dtype == "f32" else torch.int16
    k2, v2 = oracle.write_cache(
        post.k_cache.view(view).numpy(), post.v_cache.view(view).numpy(),
        post.k_new.view(view).numpy(), post.v_new.view(view).numpy(),
        post.slot_mapping.numpy(), sp.block_size,
    )
    assert np.array_equal(k2, pre.k_cache.view(view).numpy())
    assert np.array_equal(v2, pre.v_cache.view(view).numpy())
    out = oracle.decode(_np(pre.q), _np(pre.k_cache), _np(pre.v_cache), pre.block_tables.numpy(),
                        pre.context_lens.numpy(), pre.scale, sp.block_size)
    assert np.all(np.isfinite(out))


# --- multi-query (causal) ------------------------------------------------


def test_multi_query_with_one_query_is_decode():
    rng = np.random.default_rng(20)
    q, kc, vc, bt, ctx = _random_paged(rng)
    a = oracle.decode(q, kc, vc, bt, ctx, 0.3, 4)
    b = oracle.decode_multi(q[:, None], kc, vc, bt, ctx, 0.3, 4)[:, 0]
    assert np.array_equal(a, b)


def test_multi_query_matches_sdpa_with_bottom_right_causal_mask():
    """Library cross-check: torch SDPA with an explicit mask that lets query i
    (at position c - Q + i) see keys 0..c - Q + i."""
    rng = np.random.default_rng(21)
    S, Q, H, Hk, D, bs = 3, 4, 8, 2, 16, 4
    ctx = np.array([4, 9, 23])
    q4 = rng.standard_normal((S, Q, H, D))
    _, kc, vc, bt, _ = _random_paged(rng, S=S, H=H, Hk=Hk, D=D, bs=bs, max_ctx=24, nb=20, ctx=ctx)
    out = oracle.decode_multi(q4, kc, vc, bt, ctx, 0.25, bs)
    flat_k, flat_v = kc.reshape(-1, Hk, D), vc.reshape(-1, Hk, D)
    for s in range(S):
        idx = [bt[s, t // bs] * bs + t % bs for t in range(ctx[s])]
        ks = torch.from_numpy(flat_k[idx]).permute(1, 0, 2).repeat_interleave(H // Hk, 0)
        vs = torch.from_numpy(flat_v[idx]).permute(1, 0, 2).repeat_interleave(H // Hk, 0)
        qs = torch.from_numpy(q4[s]).permute(1, 0, 2)  # [H, Q, D]
        pos = torch.arange(ctx[s] - Q, ctx[s])[:, None]
        mask = torch.arange(ctx[s])[None, :] <= pos  # [Q, ctx]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=0.25)
        np.testing.assert_allclose(out[s], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-13)


def test_multi_query_prefix_consistency_and_short_context():
    """Query i equals a one-query decode over the first c - Q + i + 1 tokens;
    queries whose position is negative give zeros."""
    rng = np.random.default_rng(22)
    q, kc, vc, bt, _ = _random_paged(rng, S=2, max_ctx=23, ctx=[2, 17])
    Q = 3
    q3 = rng.standard_normal((2, Q, q.shape[1], q.shape[2]))
    ctx = np.array([2, 17])
    out = oracle.decode_multi(q3, kc, vc, bt, ctx, 0.4, 4)
    assert np.all(out[0, 0] == 0)  # position -1
    for s in range(2):
        for i in range(Q):
            pos = ctx[s] - Q + i
            if pos < 0:
                continue
            one = oracle.decode(q3[:, i], kc, vc, bt, np.array([pos + 1] * 2), 0.4, 4)[s]
            np.testing.assert_allclose(out[s, i], one, rtol=0, atol=1e-13)


# --- fp8 (E4M3) quantised cache ------------------------------------------

from oracle import fp8 as ofp8  # noqa: E402


def test_e4m3_code_table_landmarks():
    """Values fixed by the format: bias 7, 3 mantissa bits, max 448, min subnormal 2^-9."""
    d = ofp8.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0x7F, 0xFE, 0x80]))
    assert list(d[:6]) == [0.0, 2.0**-9, 7 * 2.0**-9, 2.0**-6, 1.0, 448.0]
    assert np.isnan(d[6]) and d[7] == -448.0 and d[8] == 0.0


def test_e4m3_round_trip_and_ties_to_even():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], dtype=np.uint8)
    assert np.array_equal(ofp8.e4m3_encode(ofp8.e4m3_decode(codes)), codes)
    assert ofp8.e4m3_encode([-0.0, -1e-6])[0] == 0x80 and ofp8.e4m3_encode([-1e-6])[0] == 0x80
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (001): the even one.
    assert ofp8.e4m3_encode([1.0625])[0] == 0x38
    assert ofp8.e4m3_encode([1.1875])[0] == 0x3A  # between 001 and 010 -> 010
    assert ofp8.e4m3_encode([1000.0, -1e9])[0] == 0x7E and ofp8.e4m3_encode([-1e9])[0] == 0xFE


def test_e4m3_matches_torch_in_range():
    """Library cross-check inside the finite range (torch gives NaN beyond 448,
    where the reading saturates instead)."""
    rng = np.random.default_rng(30)
    x = np.concatenate([rng.standard_normal(20000) * 4, rng.uniform(-448, 448, 2000), rng.standard_normal(2000) * 1e-3])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ofp8.e4m3_encode(x.astype(np.float32).astype(np.float64)), ref)


def test_fp8_decode_is_decode_of_dequantised_pool():
    rng = np.random.default_rng(31)
    q, kc, vc, bt, ctx = _random_paged(rng)
    kcode = ofp8.e4m3_encode(kc / 0.5)
    vcode = ofp8.e4m3_encode(vc / 0.25)
    out = ofp8.decode_fp8(q, kcode, vcode, bt, ctx, 0.3, 4, 0.5, 0.25)
    ref = oracle.decode(q, ofp8.e4m3_decode(kcode) * 0.5, ofp8.e4m3_decode(vcode) * 0.25, bt, ctx, 0.3, 4)
    assert np.array_equal(out, ref)
    # Quantisation error stays within half an E4M3 step of the scaled values.
    assert np.max(np.abs(ofp8.e4m3_decode(kcode) * 0.5 - kc)) <= 0.5 * 0.5 * 2.0**-3 * np.max(np.abs(kc)) * 2


# --- the quantiser: code of x / scale, quotient in fp32 ------------------------
#
# The pages name quantised KV caches without a format; the reading is E4M3 codes
# with one fp32 scale per pool, each code the nearest to the fp32 quotient
# x / scale.  These pins hold `quantize` and `write_cache_fp8` to facts that
# do not go through them: hand-derived codes, the fp32/exact quotient split at
# tie points, torch's own E4M3 cast of the fp32 quotient, and the scatter's
# byte-for-byte locality.  A quantiser that multiplies by the scale, divides in
# fp64, or loses the sign of a zero fails at least one of them.


def _f32(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def test_quantize_hand_derived_codes():
    # 100 / 4 = 25 = 16 * 1.5625: halfway between 1.5 (mantissa 100) and 1.625
    # (101), ties to the even mantissa: 24 = exponent field 4 + 7 = 1011, code
    # 0 1011 100.  (100 * 4 = 400 would give 384, code 0x7C.)
    assert ofp8.quantize(np.array([100.0]), 4.0)[0] == 0x5C
    # 1000 / 4 = 250 lies between 240 (0x77) and 256 (0x78) and is nearer 256.
    # (1000 * 4 saturates to 448, code 0x7E.)
    assert ofp8.quantize(np.array([1000.0]), 4.0)[0] == 0x78
    # Saturation keeps the sign: -1e6 / 0.5 -> -448.
    assert ofp8.quantize(np.array([-1e6]), 0.5)[0] == 0xFE
    # 3 / 0.75 = 4 exactly (2^2: exponent field 9 = 1001, mantissa 000).
    assert ofp8.quantize(np.array([3.0]), 0.75)[0] == 0x48


def test_quantize_keeps_the_sign_of_zero():
    # Quotients that round to zero keep the input's sign bit, as IEEE rounding
    # does: -0 -> 0x80, a negative value below half the smallest subnormal
    # (2^-10) -> 0x80, a positive one -> 0x00.
    codes = ofp8.quantize(np.array([-0.0, -1e-30, -2.0**-12, 0.0, 1e-30, 2.0**-12]), 2.0)
    assert list(codes) == [0x80, 0x80, 0x80, 0x00, 0x00, 0x00]


def test_quantize_power_of_two_scales_are_exact_reciprocals():
    # Dividing by 2^k is exact in fp32 (no overflow or underflow here), so the
    # code is the encoder's code of x * 2^-k, whatever the rounding precision.
    rng = np.random.default_rng(40)
    x = (rng.standard_normal(5000) * 30).astype(np.float32)
    for k in (-3, -1, 0, 2, 5):
        s = 2.0**k
        want = ofp8.e4m3_encode(x.astype(np.float64) * 2.0**-k)
        assert np.array_equal(ofp8.quantize(x, s), want), k


# fp32 pairs (x, s), as bit patterns, whose exact quotient x / s lies within
# half an fp32 ulp of an E4M3 tie point (the midpoint of two neighbouring
# codes): the fp32 quotient lands exactly on the tie and rounds to the even
# code, while the exact (or fp64) quotient is off the tie and rounds to the
# other neighbour.  Found by searching random fp32 pairs; each row re-derives
# its own premises below with exact rational arithmetic.
#   (x bits, s bits, tie point, code of the fp32 quotient, code of the exact one)
FP32_TIE_CASES = [
    # 1.0625 is halfway between 1.0 (0x38, mantissa 000) and 1.125 (0x39).
    (1071955372, 1071073562, 1.0625, 0x38, 0x39),
    (1078126519, 1077375148, 1.0625, 0x38, 0x39),
    # 1.1875 is halfway between 1.125 (0x39) and 1.25 (0x3A, mantissa 010).
    (1062307510, 1060139377, 1.1875, 0x3A, 0x39),
    (1071338826, 1069069213, 1.1875, 0x3A, 0x39),
    # 3.5 * 2^-9 is halfway between the subnormals 3 * 2^-9 (0x03) and 4 * 2^-9 (0x04).
    (1011338257, 1071929071, 0.0068359375, 0x04, 0x03),
    # Negative: -1.0625 between -1.0 (0xB8) and -1.125 (0xB9).
    (3218035470, 1069752574, -1.0625, 0xB8, 0xB9),
]


@pytest.mark.parametrize("xb, sb, tie, code32, code_exact", FP32_TIE_CASES)
def test_quantize_divides_in_fp32_at_tie_points(xb, sb, tie, code32, code_exact):
    from fractions import Fraction

    x, s = _f32(xb), _f32(sb)
    # Premises: the fp32 quotient is the tie itself, the exact one is not.
    assert float(np.float32(x) / np.float32(s)) == tie
    exact = Fraction(float(x)) / Fraction(float(s))
    assert exact != Fraction(tie)
    # The two codes are the tie's neighbours, and the exact quotient lies
    # strictly between the tie and code_exact's value, so it rounds there.
    v32, vex = ofp8.e4m3_decode(np.array([code32, code_exact], dtype=np.uint8))
    assert Fraction(tie) == (Fraction(v32) + Fraction(vex)) / 2
    assert min(Fraction(tie), Fraction(vex)) < exact < max(Fraction(tie), Fraction(vex))
    # The reading: the code is decided on the fp32 quotient.
    assert ofp8.quantize(np.array([x]), float(s))[0] == code32


def test_quantize_matches_torch_cast_of_the_fp32_quotient():
    """torch's E4M3 cast (round to nearest even from fp32) of the fp32
    quotient, for quotients inside +-448 where torch does not produce NaN."""
    rng = np.random.default_rng(41)
    x = np.concatenate([rng.standard_normal(20000) * 3, rng.uniform(-200, 200, 3000),
                        rng.standard_normal(3000) * 1e-2]).astype(np.float32)
    for s in (0.37, 1.0, 2.5, 1e-3 * 7.3, 0.0913):
        sf = np.float32(s)
        quot = x / sf
        keep = np.abs(quot) <= 448
        ref = torch.from_numpy(quot[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ofp8.quantize(x[keep], s), ref), s


def test_write_cache_fp8_scatters_torch_codes_and_nothing_else():
    rng = np.random.default_rng(42)
    nb, bs, hk, d, t = 9, 4, 2, 8, 11
    kc = rng.integers(0, 256, (nb, bs, hk, d)).astype(np.uint8)
    vc = rng.integers(0, 256, (nb, bs, hk, d)).astype(np.uint8)
    kn = (rng.standard_normal((t, hk, d)) * 2).astype(np.float32)
    vn = (rng.standard_normal((t, hk, d)) * 2).astype(np.float32)
    slots = rng.permutation(nb * bs)[:t].astype(np.int64)
    slots[[3, 7]] = -1
    ks, vs = 0.37, 2.5
    k2, v2 = ofp8.write_cache_fp8(kc, vc, kn, vn, slots, bs, ks, vs)

    def cast(a, s):
        return torch.from_numpy(a / np.float32(s)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    kwant, vwant = kc.copy(), vc.copy()
    for i, sl in enumerate(slots.tolist()):
        if sl >= 0:
            kwant[sl // bs, sl % bs] = cast(kn[i], ks)
            vwant[sl // bs, sl % bs] = cast(vn[i], vs)
    assert np.array_equal(k2, kwant) and np.array_equal(v2, vwant)
    assert k2.dtype == np.uint8
