"""Pins for the oracle's chunk of queries against a paged cache (prefix caching /
chunked prefill; yapayzekasozluk.tr "attention" tag page, entry "KV Cache").
Checked against the decode and dense prefill entry points of the oracle, which
are separate code paths: a one-query chunk is a decode step, and a chunk is
the last rows of causal prefill over the whole sequence."""
import numpy as np

from attn_fwd_07_b300 import inputs


def dense_of(c, b):
    """Sequence b's cached keys/values as dense [1, n, Hkv, d] float32 arrays."""
    n = int(c.seq_lens[b])
    pt = c.page_table.numpy()
    kc, vc = c.k_cache.float().numpy(), c.v_cache.float().numpy()
    k = np.stack([kc[pt[b, t // 16], t % 16] for t in range(n)])[None]
    v = np.stack([vc[pt[b, t // 16], t % 16] for t in range(n)])[None]
    return k, v


def test_one_query_chunk_is_a_decode_step(oracle):
    """q_len = 1: the query sits at the newest position and sees every cached token,
    which is the paged decode.  Catches: an off-by-one in the query position."""
    c = inputs.chunked([1, 17, 64, 300], [1, 1, 1, 1], 8, 2, 16, 41)
    o, lse = oracle.chunk_paged_rows(c.q.float().numpy(), c.k_cache.float().numpy(),
                                     c.v_cache.float().numpy(), c.page_table.numpy(),
                                     c.seq_lens.numpy(), c.cu_seqlens_q.numpy(), True, c.scale)
    od, ld = oracle.decode_paged(c.q.float().numpy(), c.k_cache.float().numpy(),
                                 c.v_cache.float().numpy(), c.page_table.numpy(),
                                 c.seq_lens.numpy(), c.scale)
    np.testing.assert_array_equal(o.reshape(od.shape), od)
    np.testing.assert_array_equal(lse.reshape(ld.shape), ld)


def test_chunk_is_the_tail_of_causal_prefill(oracle):
    """The chunk's queries are the last q_len rows of causal prefill over the whole
    sequence (any earlier query rows), including a chunk that is the whole sequence.
    Catches: a wrong causal offset, the wrong page of a key, a wrong head map."""
    ctx, ql = [40, 100, 33, 16], [7, 100, 1, 16]
    c = inputs.chunked(ctx, ql, 4, 2, 8, 42)
    o, lse = oracle.chunk_paged_rows(c.q.float().numpy(), c.k_cache.float().numpy(),
                                     c.v_cache.float().numpy(), c.page_table.numpy(),
                                     c.seq_lens.numpy(), c.cu_seqlens_q.numpy(), True, c.scale)
    o = o.reshape(-1, 4, 8)
    lse = lse.reshape(-1, 4)
    cu = c.cu_seqlens_q.numpy()
    rng = np.random.default_rng(0)
    for b, (n, m) in enumerate(zip(ctx, ql)):
        k, v = dense_of(c, b)
        qd = rng.standard_normal((1, n, 4, 8)).astype(np.float32)
        qd[0, n - m:] = c.q.float().numpy()[cu[b]:cu[b + 1]]
        od, ld = oracle.attn_fwd(qd, k, v, True, c.scale)
        np.testing.assert_allclose(o[cu[b]:cu[b + 1]], od[0, n - m:], rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse[cu[b]:cu[b + 1]], ld[0, :, n - m:].T, rtol=0, atol=1e-13)


def test_non_causal_chunk_rows_are_decode_steps(oracle):
    """Without the causal rule every chunk query sees all cached tokens: each row
    equals a decode step with that query."""
    c = inputs.chunked([50, 70], [5, 3], 4, 4, 8, 43, causal=False)
    o, lse = oracle.chunk_paged_rows(c.q.float().numpy(), c.k_cache.float().numpy(),
                                     c.v_cache.float().numpy(), c.page_table.numpy(),
                                     c.seq_lens.numpy(), c.cu_seqlens_q.numpy(), False, c.scale)
    o = o.reshape(-1, 4, 8)
    lse = lse.reshape(-1, 4)
    cu = c.cu_seqlens_q.numpy()
    for b in range(2):
        for t in range(cu[b], cu[b + 1]):
            qd = c.q.float().numpy()[t][None].repeat(2, 0)
            od, ld = oracle.decode_paged(qd, c.k_cache.float().numpy(), c.v_cache.float().numpy(),
                                         c.page_table.numpy(), c.seq_lens.numpy(), c.scale,
                                         seqs=[b])
            np.testing.assert_allclose(o[t], od[0], rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[t], ld[0], rtol=0, atol=1e-13)
