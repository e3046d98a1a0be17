"""Pins for the fp64 oracle: checks against what the attention pages and plain
mathematics fix, none of which re-runs the oracle's own formula.

Sources:
* "Donanıma Duyarlı Algoritma Tasarımı: FlashAttention" (fatihsoysal.com):
  section "Transformer Mimarisi ve Self-Attention Mekanizması" (the attention
  formula and the row-wise softmax), section "FlashAttention'ın Temelleri"
  (softmax(x) = softmax(x - c)), section "Online Softmax Prensibi" (steps 1-5).
* yapayzekasozluk.tr "attention" tag page, entry "KV Cache" (cached keys and
  values, grouped query heads sharing key/value heads, fixed-size pages).

Each test names the plausible oracle mistakes it would catch.
"""
import json
import math
import os
from fractions import Fraction

import mpmath
import numpy as np
import pytest
from scipy.special import expit

from attn_fwd_07_b300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


# ---------------------------------------------------------------- closed forms

def test_single_key_returns_v(oracle):
    """N=1: the softmax over one key is 1, so O = V[0] and LSE = s_00.
    Catches: a missing normalisation, a LSE without the max term."""
    q, k, v = rnd((2, 1, 3, 8), 1), rnd((2, 1, 3, 8), 2), rnd((2, 1, 3, 8), 3)
    scale = 0.37
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, scale)
        np.testing.assert_array_equal(o, v.astype(np.float64))
        s00 = scale * np.einsum("bnhd,bnhd->bhn", q.astype(np.float64), k.astype(np.float64))
        np.testing.assert_allclose(lse, s00, rtol=0, atol=1e-14)


def test_identical_keys_give_mean_of_values(oracle):
    """All keys equal: every score in a row is the same s, so O = mean of the V
    rows and LSE = s + ln N.  Catches: weights not summing to one, an O that
    divides by the wrong sum, a dropped ln N."""
    B, N, H, d = 1, 37, 2, 16
    q = rnd((B, N, H, d), 4)
    k = np.repeat(rnd((B, 1, H, d), 5), N, axis=1)
    v = rnd((B, N, H, d), 6)
    scale = 0.25
    o, lse = oracle.attn_fwd(q, k, v, False, scale)
    mean_v = v.astype(np.float64).mean(axis=1, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean_v, o.shape), rtol=0, atol=1e-13)
    s = scale * np.einsum("bnhd,bhd->bhn", q.astype(np.float64), k[:, 0].astype(np.float64))
    np.testing.assert_allclose(lse, s + math.log(N), rtol=0, atol=1e-12)


def test_causal_row0_is_v0(oracle):
    """Causal: query 0 sees only key 0, so O[0] = V[0] exactly and LSE = s_00.
    Catches: the mask off by one, the mask applied to the wrong axis."""
    q, k, v = rnd((3, 20, 2, 8), 7), rnd((3, 20, 2, 8), 8), rnd((3, 20, 2, 8), 9)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.5)
    np.testing.assert_array_equal(o[:, 0], v[:, 0].astype(np.float64))
    s00 = 0.5 * np.einsum("bhd,bhd->bh", q[:, 0].astype(np.float64), k[:, 0].astype(np.float64))
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-14)


def test_zero_query_gives_prefix_means(oracle):
    """Q = 0: all scores are 0, so non-causal O = mean(V), LSE = ln N, and causal
    row i = mean(V[0..i]), LSE = ln(i+1).  Catches: a causal mask that keeps
    j < i or j <= i+1, a wrong count in the denominator."""
    B, N, H, d = 2, 50, 1, 4
    q = np.zeros((B, N, H, d), np.float32)
    k, v = rnd((B, N, H, d), 10), rnd((B, N, H, d), 11)
    o, lse = oracle.attn_fwd(q, k, v, False, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.astype(np.float64).mean(1, keepdims=True),
                                                  o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-14)
    o, lse = oracle.attn_fwd(q, k, v, True, 1.0)
    prefix = np.cumsum(v.astype(np.float64), axis=1) / np.arange(1, N + 1)[None, :, None, None]
    np.testing.assert_allclose(o, prefix, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1))[None, None, :]
                               * np.ones((B, H, 1)), atol=1e-14)


def test_two_keys_reduce_to_the_logistic_function(oracle):
    """Two keys: the softmax weight of key 0 is the logistic function of
    s_0 - s_1 and the LSE is log(exp s_0 + exp s_1) (scipy's expit and numpy's
    logaddexp).  Catches: a dropped or inverted scale, a sign error, P V taken
    with the weights of the other key."""
    d = 8
    q, k, v = rnd((1, 2, 1, d), 12), rnd((1, 2, 1, d), 13, 2.0), rnd((1, 2, 1, d), 14)
    for scale in (0.125, 0.5, 2.0):
        o, lse = oracle.attn_fwd(q, k, v, False, scale)
        q64, k64, v64 = (a[0, :, 0].astype(np.float64) for a in (q, k, v))
        for i in range(2):
            s0, s1 = scale * q64[i] @ k64[0], scale * q64[i] @ k64[1]
            w0 = expit(s0 - s1)
            np.testing.assert_allclose(o[0, i, 0], w0 * v64[0] + (1 - w0) * v64[1],
                                       rtol=1e-13, atol=1e-14)
            assert abs(lse[0, 0, i] - np.logaddexp(s0, s1)) < 1e-13


def test_rows_are_distributions_and_shift_invariant(oracle):
    """With V = identity (d = N), O is the probability matrix P itself: its rows
    are non-negative and sum to 1.  Appending a coordinate that adds the same
    constant c to every score of every row (q extra = 1, k extra = c/scale)
    leaves O unchanged and moves LSE by exactly c: softmax(x) = softmax(x - c).
    Catches: an unnormalised P, a max shift that changes the result."""
    N = 12
    q = rnd((1, N, 1, N), 15)
    k = rnd((1, N, 1, N), 16)
    v = np.eye(N, dtype=np.float32)[None, :, None, :]
    for causal in (False, True):
        P, lse = oracle.attn_fwd(q, k, v, causal, 0.6)
        P = P[0, :, 0, :]
        assert (P >= 0).all()
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        if causal:
            assert np.all(np.triu(P, 1) == 0)
        c = 7.5
        q2 = np.concatenate([q, np.ones((1, N, 1, 1), np.float32)], axis=3)
        k2 = np.concatenate([k, np.full((1, N, 1, 1), c / 0.6, np.float32)], axis=3)
        # c / 0.6 is rounded to fp32: the exact shift is 0.6 * fl32(c / 0.6)
        shift = 0.6 * float(np.float32(c / 0.6))
        v2 = np.concatenate([v, np.zeros((1, N, 1, 1), np.float32)], axis=3)
        P2, lse2 = oracle.attn_fwd(q2, k2, v2, causal, 0.6)
        np.testing.assert_allclose(P2[0, :, 0, :N], P, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse + shift, rtol=0, atol=1e-12)


def test_large_scores_do_not_overflow(oracle):
    """Scores of several hundred: exp(s) alone would overflow fp64 past ~709;
    the max shift keeps the oracle finite, and a row whose top score beats the
    rest by far puts all its weight on that key."""
    d = 4
    q = np.zeros((1, 3, 1, d), np.float32)
    q[0, :, 0, 0] = 100.0
    k = np.zeros((1, 3, 1, d), np.float32)
    k[0, :, 0, 0] = [10.0, 9.0, 1.0]
    v = rnd((1, 3, 1, d), 17)
    o, lse = oracle.attn_fwd(q, k, v, False, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(o[0, :, 0], np.broadcast_to(v[0, 0, 0], (3, d)), atol=1e-40)
    np.testing.assert_allclose(lse, 1000.0 + math.log1p(math.exp(-100.0) + math.exp(-900.0)),
                               rtol=1e-15)


# ---------------------------------------------------------------- worked examples

def _frac(x):
    return float(Fraction(x))


def test_golden_integer_log_scores(oracle):
    """Hand-derived example (tests/golden/integer_log_scores.json): scores j ln 2
    give weights 2^j / (2^n - 1)."""
    g = json.load(open(os.path.join(GOLDEN, "integer_log_scores.json")))
    q = np.array(g["q"], np.float32)[None, :, None, :]
    k = np.array(g["k"], np.float32)[None, :, None, :]
    v = np.array(g["v"], np.float32)[None, :, None, :]
    for mode, causal in (("noncausal", False), ("causal", True)):
        o, lse = oracle.attn_fwd(q, k, v, causal, math.log(2.0))
        want_o = np.array([[_frac(x) for x in row] for row in g[mode]["o"]])
        want_lse = np.array([math.log(_frac(x)) for x in g[mode]["lse_of"]])
        np.testing.assert_allclose(o[0, :, 0], want_o, rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(lse[0, 0], want_lse, rtol=0, atol=1e-14)


def test_golden_online_softmax_blocks(oracle):
    """Hand-derived run of the pages' online recurrence
    (tests/golden/online_softmax_blocks.json): (M, L) after each block."""
    g = json.load(open(os.path.join(GOLDEN, "online_softmax_blocks.json")))
    x = np.array(g["x_log2"], np.float64) * math.log(2.0)
    blk = g["block"]
    for nb, want in enumerate(g["after_each_block"], start=1):
        M, L = oracle.online_softmax_stats(x[:nb * blk], blk)
        assert abs(M - want["M_log2"] * math.log(2.0)) < 1e-15
        assert abs(L - _frac(want["L"])) < 1e-15


# ---------------------------------------------------------------- brute force

def _brute(q, k, v, causal, scale, group):
    """50-digit evaluation of the formula with no max shift: O = sum exp(s) v / sum exp(s)."""
    mpmath.mp.dps = 50
    B, N, Hq, d = q.shape
    o = np.zeros(q.shape, np.float64)
    lse = np.zeros((B, Hq, N), np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(N):
                n = i + 1 if causal else N
                e = []
                for j in range(n):
                    s = mpmath.mpf(0)
                    for c in range(d):
                        s += mpmath.mpf(float(q[b, i, h, c])) * mpmath.mpf(float(k[b, j, g, c]))
                    e.append(mpmath.exp(mpmath.mpf(scale) * s))
                Z = mpmath.fsum(e)
                for c in range(d):
                    o[b, i, h, c] = float(mpmath.fsum(e[j] * mpmath.mpf(float(v[b, j, g, c]))
                                                      for j in range(n)) / Z)
                lse[b, h, i] = float(mpmath.log(Z))
    return o, lse


@pytest.mark.parametrize("B,N,Hq,Hkv,d,causal", [
    (1, 5, 1, 1, 3, False), (2, 7, 2, 1, 4, True), (1, 8, 4, 2, 2, True), (1, 6, 3, 3, 4, False),
])
def test_brute_force_tiny(oracle, B, N, Hq, Hkv, d, causal):
    """Tiny random shapes against a 50-digit evaluation of the formula without the
    max shift.  Catches: a transposed operand, a wrong head map, a wrong index
    anywhere, a wrong scale."""
    seed = B * 1000 + N * 100 + Hq * 10 + d
    q, k, v = rnd((B, N, Hq, d), seed), rnd((B, N, Hkv, d), seed + 1), rnd((B, N, Hkv, d), seed + 2)
    scale = 0.7
    o, lse = oracle.attn_fwd(q, k, v, causal, scale)
    ob, lb = _brute(q, k, v, causal, scale, Hq // Hkv)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- structure

def test_gqa_equals_mha_with_repeated_kv_heads(oracle):
    """Grouped query heads h use kv head h // (Hq/Hkv): the result equals plain
    multi-head attention with each kv head repeated for its group.  Catches: the
    h % Hkv map, groups of the wrong size."""
    B, N, Hq, Hkv, d = 2, 33, 8, 2, 8
    q, k, v = rnd((B, N, Hq, d), 20), rnd((B, N, Hkv, d), 21), rnd((B, N, Hkv, d), 22)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.3)
        kr, vr = np.repeat(k, Hq // Hkv, axis=2), np.repeat(v, Hq // Hkv, axis=2)
        o2, lse2 = oracle.attn_fwd(q, kr, vr, causal, 0.3)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
    # and a kv head's value change only moves its own query group
    # (doubling is exact in binary floating point, and O is linear in V)
    v3 = v.copy()
    v3[:, :, 1] *= 2.0
    o3, _ = oracle.attn_fwd(q, k, v3, False, 0.3)
    o, _ = oracle.attn_fwd(q, k, v, False, 0.3)
    np.testing.assert_array_equal(o3[:, :, :4], o[:, :, :4])
    np.testing.assert_array_equal(o3[:, :, 4:], 2.0 * o[:, :, 4:])


def test_varlen_equals_per_sequence_dense(oracle):
    """Packed sequences are independent problems: each equals a dense call on
    its own slice (including a length-1 and an empty sequence)."""
    lens = [5, 1, 0, 17, 9]
    Hq, Hkv, d = 4, 2, 8
    w = inputs.varlen(lens, Hq, Hkv, d, seed=30, dtype=inputs.torch.float32)
    q, k, v = w.q.numpy(), w.k.numpy(), w.v.numpy()
    cu = w.cu_seqlens.numpy()
    for causal in (False, True):
        o, lse = oracle.attn_varlen(q, k, v, cu, causal, 0.4)
        for s, L in enumerate(lens):
            a, b = cu[s], cu[s + 1]
            if L == 0:
                continue
            od, ld = oracle.attn_fwd(q[None, a:b], k[None, a:b], v[None, a:b], causal, 0.4)
            np.testing.assert_array_equal(o[a:b], od[0])
            np.testing.assert_array_equal(lse[:, a:b], ld[0])


def test_empty_rows_are_zero_with_minus_inf_lse(oracle):
    """A query with no keys (rows of a zero-length problem, never reached by a
    non-empty one): O = 0 and LSE = -inf by the stated convention."""
    q = rnd((1, 3, 1, 4), 31)
    k = np.zeros((1, 0, 1, 4), np.float32)
    o, lse = oracle.attn_rows(q, k, k, [[0, 0, 0], [0, 0, 2]], False, 1.0)
    assert (o == 0).all() and np.isneginf(lse).all()


def _contiguous_reference(oracle, w, b, scale):
    """Sequence b's cache gathered in logical order and run as a one-query dense problem."""
    L = int(w.seq_lens[b])
    ps = w.page_size
    pages = w.page_table[b, :(L + ps - 1) // ps].numpy()
    kc, vc = w.k_cache.numpy(), w.v_cache.numpy()
    K = kc[pages].reshape(-1, kc.shape[2], kc.shape[3])[:L]
    V = vc[pages].reshape(-1, vc.shape[2], vc.shape[3])[:L]
    q = w.q.numpy()[b][None, None]          # [1, 1, Hq, d]
    return oracle.attn_rows(q, K[None], V[None],
                            [[0, h, 0] for h in range(q.shape[2])], False, scale)


def test_decode_paged_equals_contiguous_and_is_permutation_invariant(oracle):
    """Paged cache = contiguous cache behind a page table: the decode result
    equals one query attending to the gathered keys in logical order, and
    renumbering the physical pages (with the table) changes nothing.  Lengths
    cover 1, a partial page, exactly one page and several pages."""
    lens = [1, 15, 16, 17, 40]
    w = inputs.paged(lens, 4, 2, 8, seed=40, page_size=16, max_pages=4,
                     dtype=inputs.torch.float32)
    o, lse = oracle.decode_paged(w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens, 0.35)
    for b in range(len(lens)):
        oc, lc = _contiguous_reference(oracle, w, b, 0.35)
        np.testing.assert_array_equal(o[b], oc)
        np.testing.assert_array_equal(lse[b], lc)
    P = w.k_cache.shape[0]
    perm = np.random.default_rng(41).permutation(P)
    inv = np.argsort(perm)        # new id of old page p is inv[p]
    kc2 = w.k_cache.numpy()[perm]
    vc2 = w.v_cache.numpy()[perm]
    pt = w.page_table.numpy()
    pt2 = np.where(pt >= 0, inv[np.maximum(pt, 0)], -1).astype(np.int32)
    o2, lse2 = oracle.decode_paged(w.q, kc2, vc2, pt2, w.seq_lens, 0.35)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_decode_equals_last_causal_prefill_row(oracle):
    """The new token of decode sees every cached token, which is what the last
    row of causal prefill over the same keys sees."""
    N, Hq, Hkv, d = 37, 4, 2, 8
    q, k, v = rnd((1, N, Hq, d), 50), rnd((1, N, Hkv, d), 51), rnd((1, N, Hkv, d), 52)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.45)
    ps = 8
    npg = (N + ps - 1) // ps
    kc = np.zeros((npg, ps, Hkv, d), np.float32)
    vc = np.zeros((npg, ps, Hkv, d), np.float32)
    kc.reshape(-1, Hkv, d)[:N] = k[0]
    vc.reshape(-1, Hkv, d)[:N] = v[0]
    pt = np.arange(npg, dtype=np.int32)[None]
    od, ld = oracle.decode_paged(q[:, N - 1], kc, vc, pt, np.array([N], np.int32), 0.45)
    np.testing.assert_allclose(od[0], o[0, N - 1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(ld[0], lse[0, :, N - 1], rtol=0, atol=1e-15)


def test_decode_rejects_bad_page_ids(oracle):
    lens = [20]
    w = inputs.paged(lens, 2, 1, 4, seed=60, page_size=16, dtype=inputs.torch.float32)
    pt = w.page_table.clone()
    pt[0, 1] = w.k_cache.shape[0]
    with pytest.raises(ValueError):
        oracle.decode_paged(w.q, w.k_cache, w.v_cache, pt, w.seq_lens, 1.0)


# ---------------------------------------------------------------- recurrence

@pytest.mark.parametrize("block", [1, 3, 16, 64, 1000])
def test_online_recurrence_reaches_direct_max_and_sum(oracle, block):
    """Steps 1-5 of the online softmax, run block by block, end at the direct
    max and sum exp(x - max) for any block size."""
    x = np.random.default_rng(70).standard_normal(777) * 6.0
    M, L = oracle.online_softmax_stats(x, block)
    m = x.max()
    assert M == m
    assert abs(L - math.fsum(np.exp(x - m))) <= 1e-12 * L


def test_split_and_merge_equals_attention_over_all_keys(oracle):
    """Attention over disjoint key chunks, combined by their log-sum-exps, equals
    attention over all keys (the rule the split decode uses)."""
    N, d = 300, 16
    q, k, v = rnd((1, 1, 1, d), 80), rnd((1, N, 1, d), 81), rnd((1, N, 1, d), 82)
    o_all, lse_all = oracle.attn_rows(q, k, v, [[0, 0, 0]], False, 0.5)
    for cuts in ([0, 300], [0, 1, 300], [0, 100, 200, 300], [0, 7, 7, 150, 299, 300]):
        parts_o, parts_l = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o_s, l_s = oracle.attn_rows(q, k[:, a:b], v[:, a:b], [[0, 0, 0]], False, 0.5)
            parts_o.append(o_s[0])
            parts_l.append(l_s[0])
        o_m, l_m = oracle.merge_parts(np.stack(parts_o), np.array(parts_l))
        np.testing.assert_allclose(o_m, o_all[0], rtol=0, atol=1e-13)
        assert abs(l_m - lse_all[0]) < 1e-12


def test_rows_entry_matches_full_entry(oracle):
    """The row-sampling entry returns exactly the full entry's rows."""
    q, k, v = rnd((2, 19, 4, 8), 90), rnd((2, 19, 2, 8), 91), rnd((2, 19, 2, 8), 92)
    o, lse = oracle.attn_fwd(q, k, v, True, 0.3)
    rows = [[1, 3, 18], [0, 0, 0], [1, 1, 7]]
    orow, lrow = oracle.attn_rows(q, k, v, rows, True, 0.3)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(orow[r], o[b, i, h])
        assert lrow[r] == lse[b, h, i]
