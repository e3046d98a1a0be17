"""GPU parity for a chunk of queries against a paged cache (attn_fwd_chunked_paged)
against the fp64 oracle on the same seeded inputs: chunks of 1 to a whole
sequence, ragged tails, prefixes shorter and longer than a key tile, both CTA
pairings, causal and not, a bad page id and invalid sizes (reported, never
read), agreement with the dense causal prefill on a contiguous page table, and
the 8-sequence workload on sampled rows.  Tolerances are in tests/parity.py."""
import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    assert A.attn_get_device_status() == 0


def f32(t):
    return t.float().cpu().numpy()


def check_status():
    st = A.attn_get_device_status()
    assert st == 0, A.attn_status_string(st)


def run(c, page_table=None, seq_lens=None):
    pt = c.page_table if page_table is None else page_table
    sl = c.seq_lens if seq_lens is None else seq_lens
    return A.attn_fwd_chunked_paged(c.q.cuda(), c.k_cache.cuda(), c.v_cache.cuda(), pt.cuda(),
                                    sl.cuda(), c.cu_seqlens_q.cuda(), int(c.q_lens.max()),
                                    c.causal, c.scale)


def ref(oracle, c, rows=None):
    return oracle.chunk_paged_rows(f32(c.q), f32(c.k_cache), f32(c.v_cache),
                                   c.page_table.numpy(), c.seq_lens.numpy(),
                                   c.cu_seqlens_q.numpy(), c.causal, c.scale, rows=rows)


def compare(o, lse, o_ref, lse_ref, Hq, what):
    og = f32(o).reshape(-1, o.shape[-1])
    lg = f32(lse).T.reshape(-1)  # [Hq, Tq] -> rows (t, h) in t-major order
    assert_close(errors(og, o_ref, lg, lse_ref), what)


CHUNK_CASES = [
    # ctx_lens, q_lens, Hq, Hkv, d, causal
    ([1], [1], 2, 1, 128, True), ([300, 17], [300, 1], 4, 2, 128, True),
    ([1000, 129, 2048], [77, 129, 256], 8, 2, 128, True), ([640, 300], [128, 255], 3, 3, 64, True),
    ([513, 40], [200, 40], 4, 4, 128, False), ([4096], [1000], 32, 8, 128, True),
    ([2000, 2000], [1, 1999], 2, 2, 64, True),
]


@pytest.mark.parametrize("ctx,ql,Hq,Hkv,d,causal", CHUNK_CASES)
def test_chunk_small(oracle, ctx, ql, Hq, Hkv, d, causal):
    c = inputs.chunked(ctx, ql, Hq, Hkv, d, 6000 + sum(ctx) + sum(ql) + Hq + d, causal=causal)
    o, lse = run(c)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = ref(oracle, c)
    compare(o, lse, o_ref, lse_ref, Hq, (ctx, ql, Hq, Hkv, d, causal))


def test_whole_sequence_chunk_equals_causal_prefill():
    """A chunk that is the whole sequence, with pages in order, is causal prefill: the
    same result as attn_fwd_varlen over the same tokens laid out contiguously."""
    ctx = [700, 333]
    c = inputs.chunked(ctx, ctx, 8, 2, 128, 6100)
    pt = torch.full_like(c.page_table, -1)
    kd, vd = [], []
    npg = 0
    for b, n in enumerate(ctx):
        pages = c.page_table[b, :(n + 15) // 16]
        kd.append(c.k_cache[pages.long()].reshape(-1, 2, 128)[:n])
        vd.append(c.v_cache[pages.long()].reshape(-1, 2, 128)[:n])
        npg += len(pages)
    o1, l1 = run(c)
    k = torch.cat(kd).cuda()
    v = torch.cat(vd).cuda()
    o2, l2 = A.attn_fwd_varlen(c.q.cuda(), k, v, c.cu_seqlens_q.cuda(), max(ctx), True, c.scale)
    torch.cuda.synchronize()
    check_status()
    e = errors(f32(o1), f32(o2), f32(l1), f32(l2))
    assert e["max_o"] <= 1e-2 and e["max_lse"] <= 1e-4, e


def test_chunk_bad_page_id_is_reported(oracle):
    c = inputs.chunked([300, 300], [100, 100], 4, 2, 128, 6200)
    pt = c.page_table.clone()
    pt[1, 3] = -5
    o, lse = run(c, page_table=pt)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BOUNDS
    # sequence 0 does not touch the bad entry
    rows = np.stack(np.meshgrid(np.arange(100), np.arange(4), indexing="ij"), -1).reshape(-1, 2)
    o_ref, lse_ref = ref(oracle, c, rows=rows)
    compare(o[:100], lse[:, :100], o_ref, lse_ref, 4, "sequence 0")


def test_chunk_longer_than_cache_is_reported_and_skipped():
    c = inputs.chunked([64], [64], 2, 2, 128, 6300)
    o, lse = run(c, seq_lens=torch.tensor([32], dtype=torch.int32))
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BOUNDS


def test_workload_chunked_prefill_sampled(oracle):
    """8 sequences, cached prefixes U[1024,16384] + 2048-token chunks (as the benchmark
    runs it): sampled rows of every sequence, chunk ends included."""
    c = inputs.make("chunked_prefill_b8")
    o, lse = run(c)
    torch.cuda.synchronize()
    check_status()
    cu = c.cu_seqlens_q.numpy()
    rng = np.random.default_rng(7)
    t = np.concatenate([cu[:-1], cu[1:] - 1, rng.integers(0, cu[-1], 240)])
    h = rng.integers(0, 32, len(t))
    rows = np.stack([t, h], 1)
    o_ref, lse_ref = ref(oracle, c, rows=rows)
    og = f32(o)[t, h]
    lg = f32(lse)[h, t]
    assert_close(errors(og, o_ref, lg, lse_ref), "chunked_prefill_b8")
