"""Pins for the oracle's sliding-window attention (yapayzekasozluk.tr "attention"
tag page, entry "Sliding Window Attention": each token attends only to the
tokens within w/2 of its own position on either side instead of the whole
sequence).  Checked against closed forms, the full and causal oracle entry
points (independent code paths), and a 50-digit brute force; none re-runs the
window routine's own formula.
"""
import math

import mpmath
import numpy as np
import pytest


def rnd(shape, seed, scale=1.0):
    return (np.random.default_rng(seed).standard_normal(shape) * scale).astype(np.float32)


def test_zero_window_attends_only_to_itself(oracle):
    """wl = wr = 0: the only key of row i is key i, so O = V[i] and LSE = s_ii.
    Catches: an off-by-one in either bound, a wrong key offset."""
    B, N, Hq, Hkv, d = 2, 11, 4, 2, 8
    q, k, v = rnd((B, N, Hq, d), 1), rnd((B, N, Hkv, d), 2), rnd((B, N, Hkv, d), 3)
    o, lse = oracle.attn_window(q, k, v, 0, 0, 0.4)
    vr = np.repeat(v.astype(np.float64), Hq // Hkv, axis=2)
    kr = np.repeat(k.astype(np.float64), Hq // Hkv, axis=2)
    np.testing.assert_array_equal(o, vr)
    s = 0.4 * np.einsum("bnhd,bnhd->bhn", q.astype(np.float64), kr)
    np.testing.assert_allclose(lse, s, rtol=0, atol=1e-14)


def test_unbounded_windows_are_full_and_causal(oracle):
    """No left limit and no right limit is full attention; no left limit and a
    zero right limit is causal attention (both from the dense entry point), and a
    window wider than the sequence changes nothing.  Catches: a bound applied on
    the wrong side, a sign error in i - wl."""
    B, N, Hq, Hkv, d = 1, 23, 2, 1, 16
    q, k, v = rnd((B, N, Hq, d), 4), rnd((B, N, Hkv, d), 5), rnd((B, N, Hkv, d), 6)
    for wl, wr, causal in ((-1, -1, False), (-1, 0, True), (N, N, False), (N + 5, 0, True),
                           (-1, N, False), (N - 1, -1, False)):
        o, lse = oracle.attn_window(q, k, v, wl, wr, 0.3)
        of, lf = oracle.attn_fwd(q, k, v, causal, 0.3)
        np.testing.assert_array_equal(o, of)
        np.testing.assert_array_equal(lse, lf)


def test_zero_query_gives_window_means(oracle):
    """Q = 0: all allowed scores are 0, so O = mean of the V rows inside the
    window [max(0, i - wl), min(N - 1, i + wr)] and LSE = ln(its size).
    Catches: a window of the wrong width, clipping at the sequence ends."""
    B, N, H, d = 1, 17, 1, 4
    q = np.zeros((B, N, H, d), np.float32)
    k, v = rnd((B, N, H, d), 7), rnd((B, N, H, d), 8)
    for wl, wr in ((3, 3), (0, 5), (6, 0), (2, 9)):
        o, lse = oracle.attn_window(q, k, v, wl, wr, 1.0)
        for i in range(N):
            lo, hi = max(0, i - wl), min(N - 1, i + wr)
            np.testing.assert_allclose(o[0, i, 0], v[0, lo:hi + 1, 0].astype(np.float64).mean(0),
                                       rtol=0, atol=1e-14)
            assert lse[0, 0, i] == pytest.approx(math.log(hi - lo + 1), abs=1e-14)


def _brute_window(q, k, v, wl, wr, scale, group):
    """50-digit evaluation with no max shift over the keys i - wl .. i + wr."""
    mpmath.mp.dps = 50
    B, N, Hq, d = q.shape
    o = np.zeros(q.shape, np.float64)
    lse = np.zeros((B, Hq, N), np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // group
            for i in range(N):
                keys = [j for j in range(N) if (wl < 0 or j >= i - wl) and (wr < 0 or j <= i + wr)]
                e = []
                for j in keys:
                    s = mpmath.fsum(mpmath.mpf(float(q[b, i, h, c])) * mpmath.mpf(float(k[b, j, g, c]))
                                    for c in range(d))
                    e.append(mpmath.exp(mpmath.mpf(scale) * s))
                Z = mpmath.fsum(e)
                for c in range(d):
                    o[b, i, h, c] = float(mpmath.fsum(e[t] * mpmath.mpf(float(v[b, j, g, c]))
                                                      for t, j in enumerate(keys)) / Z)
                lse[b, h, i] = float(mpmath.log(Z))
    return o, lse


@pytest.mark.parametrize("N,Hq,Hkv,d,wl,wr", [
    (7, 2, 1, 3, 2, 2), (9, 1, 1, 4, 1, 3), (8, 4, 2, 2, 4, 0), (6, 3, 3, 2, -1, 1),
])
def test_window_brute_force_tiny(oracle, N, Hq, Hkv, d, wl, wr):
    """Tiny random shapes against the 50-digit formula with the window written as a
    key list.  Catches: wrong bounds, wrong head map, a transposed operand."""
    seed = N * 100 + Hq * 10 + d + wl
    q, k, v = rnd((1, N, Hq, d), seed), rnd((1, N, Hkv, d), seed + 1), rnd((1, N, Hkv, d), seed + 2)
    o, lse = oracle.attn_window(q, k, v, wl, wr, 0.8)
    ob, lb = _brute_window(q, k, v, wl, wr, 0.8, Hq // Hkv)
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lb, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- windowed decode

def _paged_case(lens, Hq, Hkv, d, seed):
    from attn_fwd_07_b300 import inputs
    p = inputs.paged(lens, Hq, Hkv, d, seed, page_size=16)
    return tuple(t.float().numpy() for t in (p.q, p.k_cache, p.v_cache)) + (
        p.page_table.numpy(), p.seq_lens.numpy(), p.scale)


def test_decode_window_wide_equals_decode(oracle):
    """A window reaching back to token 0 (or -1) sees every cached token: the plain
    paged decode entry point.  Catches: a window that drops the first or last page."""
    q, kc, vc, pt, sl, sc = _paged_case([1, 17, 40, 100], 8, 2, 16, 21)
    o0, l0 = oracle.decode_paged(q, kc, vc, pt, sl, sc)
    for window in (-1, 99, 1000):
        o, l = oracle.decode_paged_window(q, kc, vc, pt, sl, window, sc)
        np.testing.assert_array_equal(o, o0)
        np.testing.assert_array_equal(l, l0)


def test_decode_window_zero_is_last_value(oracle):
    """window = 0: the query sees only the newest token, so O = its V row and
    LSE = its score.  Catches: an off-by-one at the newest token."""
    q, kc, vc, pt, sl, sc = _paged_case([1, 16, 33, 70], 4, 2, 8, 22)
    o, l = oracle.decode_paged_window(q, kc, vc, pt, sl, 0, sc)
    for b, n in enumerate(sl):
        t = n - 1
        page, slot = pt[b, t // 16], t % 16
        for h in range(4):
            g = h // 2
            np.testing.assert_array_equal(o[b, h], vc[page, slot, g].astype(np.float64))
            s = sc * float(np.dot(q[b, h].astype(np.float64), kc[page, slot, g].astype(np.float64)))
            assert l[b, h] == pytest.approx(s, abs=1e-13)


def test_decode_window_equals_last_row_of_window_prefill(oracle):
    """The windowed decode of a sequence equals the last row of windowed prefill
    (window_left = window, window_right = 0) over the same keys laid out densely.
    Catches: a window measured from the wrong end, a wrong page of the window."""
    lens = [50, 77]
    q, kc, vc, pt, sl, sc = _paged_case(lens, 4, 2, 8, 23)
    for window in (0, 5, 16, 31, 49):
        o, l = oracle.decode_paged_window(q, kc, vc, pt, sl, window, sc)
        for b, n in enumerate(sl):
            kd = np.stack([kc[pt[b, t // 16], t % 16] for t in range(n)])[None]
            vd = np.stack([vc[pt[b, t // 16], t % 16] for t in range(n)])[None]
            qd = np.zeros((1, n, 4, 8), np.float32)
            qd[0, n - 1] = q[b]
            od, ld = oracle.attn_window(qd, kd, vd, window, 0, sc)
            np.testing.assert_allclose(o[b], od[0, n - 1], rtol=0, atol=1e-14)
            np.testing.assert_allclose(l[b], ld[0, :, n - 1], rtol=0, atol=1e-13)
