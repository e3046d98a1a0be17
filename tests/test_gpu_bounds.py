"""Device-side checks of the cache and packing contracts (GPU).

The paged cache is a table of fixed-size pages (yapayzekasozluk.tr "attention" tag
page, entry "KV Cache"): seq_lens[b] may not exceed what row b of the page table can
hold, and a packed batch's cu_seqlens must start at 0, never decrease and end at the
token count.  A caller that breaks these gets ATTN_ERR_DEVICE_BOUNDS from
attn_get_device_status, the other sequences' results stay exact, and nothing is read
or written outside the buffers: every output sits between guard bands filled with a
sentinel, and the page table carries a padding row of valid page ids that a missed
length check would read (and so change the result without any other error).
"""
import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu

PAD = 4096            # guard-band elements on each side (keeps 16-byte alignment)
SENTINEL_BF16 = 1536.0   # exact in bf16
SENTINEL_F32 = -7777.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    assert A.attn_get_device_status() == 0


def f32(t):
    return t.float().cpu().numpy()


def guarded(shape, dtype, fill):
    """A device tensor of `shape` inside a larger buffer whose guard bands (and the
    tensor itself) hold `fill`; returns (view, whole buffer)."""
    n = int(np.prod(shape))
    buf = torch.full((PAD + n + PAD,), fill, dtype=dtype, device="cuda")
    return buf[PAD:PAD + n].view(shape), buf


def assert_guards_intact(buf, fill):
    head, tail = buf[:PAD].float(), buf[-PAD:].float()
    assert bool((head == fill).all()) and bool((tail == fill).all()), "guard band written"


# ---------------------------------------------------------------- paged decode

def decode_call(kind, w, o, lse, pt):
    q = w.q.cuda()
    if kind == "fp8":
        return A.attn_decode_paged_fp8(q, w.k_cache.cuda(), w.v_cache.cuda(), w.k_scale.cuda(),
                                       w.v_scale.cuda(), pt, w.seq_lens_dev, w.scale, o=o,
                                       lse=lse)
    if kind == "window":
        return A.attn_decode_paged_window(q, w.k_cache.cuda(), w.v_cache.cuda(), pt,
                                          w.seq_lens_dev, 50, w.scale, o=o, lse=lse)
    return A.attn_decode_paged(q, w.k_cache.cuda(), w.v_cache.cuda(), pt, w.seq_lens_dev,
                               w.scale, o=o, lse=lse)


def decode_oracle(oracle, kind, w, seqs, lens):
    q = f32(w.q)[seqs]
    pt = w.page_table.numpy()[seqs]
    if kind == "fp8":
        return oracle.decode_paged_fp8(q, w.k_cache.numpy(), w.v_cache.numpy(),
                                       w.k_scale.numpy(), w.v_scale.numpy(), pt, lens, w.scale)
    if kind == "window":
        return oracle.decode_paged_window(q, f32(w.k_cache), f32(w.v_cache), pt, lens, 50,
                                          w.scale)
    return oracle.decode_paged(q, f32(w.k_cache), f32(w.v_cache), pt, lens, w.scale)


@pytest.mark.parametrize("kind", ["bf16", "fp8", "window"])
def test_decode_length_past_the_page_table_is_reported_not_read(oracle, kind):
    """Sequence 1 claims one token more than its table row holds, sequence 3 a negative
    length, and the last sequence (whose row is followed only by the padding row) one
    token more as well: all three come out empty (O = 0, LSE = -inf), the others exact."""
    lens = [40, 100, 33, 70, 90]
    Hq, Hkv, d = 8, 2, 128
    maker = inputs.paged_fp8 if kind == "fp8" else inputs.paged
    w = maker(lens, Hq, Hkv, d, 5100, page_size=16)
    B, maxp = len(lens), w.page_table.shape[1]          # maxp = 7 pages (112 tokens)
    # the page table with a padding row of valid page ids after the last sequence
    pt_full = torch.zeros((B + 1, maxp), dtype=torch.int32)
    pt_full[:B] = w.page_table
    pt_full[B] = torch.arange(maxp, dtype=torch.int32) % w.k_cache.shape[0]
    pt_dev = pt_full.cuda()
    bad = [1, 3, 4]
    sl = torch.tensor(lens, dtype=torch.int32)
    sl[1] = maxp * 16 + 1
    sl[3] = -5
    sl[4] = maxp * 16 + 1
    w.seq_lens_dev = sl.cuda()
    o, obuf = guarded((B, Hq, d), torch.bfloat16, SENTINEL_BF16)
    lse, lbuf = guarded((B, Hq), torch.float32, SENTINEL_F32)
    decode_call(kind, w, o, lse, pt_dev[:B])
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BOUNDS
    assert A.attn_get_device_status() == 0
    assert_guards_intact(obuf, SENTINEL_BF16)
    assert_guards_intact(lbuf, SENTINEL_F32)
    assert torch.equal(pt_dev.cpu(), pt_full)
    for b in bad:
        assert bool((o[b].float() == 0).all()), b
        assert bool(torch.isneginf(lse[b]).all()), b
    good = [0, 2]
    o_ref, lse_ref = decode_oracle(oracle, kind, w, good, np.array([lens[b] for b in good]))
    assert_close(errors(f32(o)[good], o_ref, f32(lse)[good], lse_ref), kind)


def test_decode_length_at_the_page_table_limit_is_accepted(oracle):
    """seq_lens[b] == max_pages_per_seq * 16 exactly fills the row: no error."""
    lens = [112, 20]
    w = inputs.paged(lens, 8, 2, 128, 5101, page_size=16)
    o, lse = A.attn_decode_paged(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(),
                                 w.page_table.cuda(), w.seq_lens.cuda(), w.scale)
    assert A.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.decode_paged(f32(w.q), f32(w.k_cache), f32(w.v_cache),
                                         w.page_table.numpy(), w.seq_lens.numpy(), w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref))


# ---------------------------------------------------------------- packed prefill

def run_varlen(w, cu, total, max_seqlen, Hq):
    d = w.q.shape[2]
    o, obuf = guarded((total, Hq, d), torch.bfloat16, SENTINEL_BF16)
    lse, lbuf = guarded((Hq, total), torch.float32, SENTINEL_F32)
    A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), torch.tensor(cu, dtype=torch.int32,
                      device="cuda"), max_seqlen, True, w.scale, o=o, lse=lse)
    st = A.attn_get_device_status()
    assert_guards_intact(obuf, SENTINEL_BF16)
    assert_guards_intact(lbuf, SENTINEL_F32)
    return o, lse, st


def check_rows(oracle, w, o, lse, a, b, rows):
    """Rows `rows` (positions inside the sequence of tokens [a, b)) against the oracle."""
    q, k, v = f32(w.q), f32(w.k), f32(w.v)
    Hq = q.shape[1]
    sel = np.array([(0, h, i) for h in range(Hq) for i in rows], np.int32)
    o_ref, l_ref = oracle.attn_rows(q[None, a:b], k[None, a:b], v[None, a:b], sel, True, w.scale)
    og = f32(o)[a + sel[:, 2], sel[:, 1]]
    lg = f32(lse)[sel[:, 1], a + sel[:, 2]]
    assert_close(errors(og, o_ref, lg, l_ref), (a, b))


def untouched(o, lse, a, b):
    return (bool((o[a:b].float() == SENTINEL_BF16).all()) and
            bool((lse[:, a:b] == SENTINEL_F32).all()))


def test_varlen_sequence_longer_than_max_seqlen(oracle):
    """max_seqlen 256 sizes the launch at two 128-row tiles; the 500-token sequence gets
    its first 256 rows (exact) and the rest stays unwritten, with the error recorded."""
    lens = [100, 500, 200]
    Hq, Hkv = 4, 2
    w = inputs.varlen(lens, Hq, Hkv, 128, 5200, torch.bfloat16)
    cu = [0, 100, 600, 800]
    o, lse, st = run_varlen(w, cu, 800, 256, Hq)
    assert st == A.ATTN_ERR_DEVICE_BOUNDS
    check_rows(oracle, w, o, lse, 0, 100, range(100))
    check_rows(oracle, w, o, lse, 600, 800, range(200))
    check_rows(oracle, w, o, lse, 100, 600, [0, 1, 127, 128, 200, 255])
    assert untouched(o, lse, 356, 600)


def test_varlen_within_its_tiles_is_not_an_error(oracle):
    """A sequence a little longer than max_seqlen but inside the launch's last tile is
    computed in full: nothing is left out, so nothing is reported."""
    lens = [300, 40]
    w = inputs.varlen(lens, 4, 2, 128, 5201, torch.bfloat16)
    o, lse, st = run_varlen(w, [0, 300, 340], 340, 290, 4)
    assert st == 0
    check_rows(oracle, w, o, lse, 0, 300, [0, 255, 256, 299])


def test_varlen_decreasing_cu_seqlens(oracle):
    """cu_seqlens [0, 100, 80, 80, 300]: sequence 1 has a negative length and is skipped
    (recorded), sequence 2 is empty, sequence 3 covers tokens 80..299."""
    w = inputs.varlen([300], 4, 2, 128, 5202, torch.bfloat16)
    o, lse, st = run_varlen(w, [0, 100, 80, 80, 300], 300, 220, 4)
    assert st == A.ATTN_ERR_DEVICE_BOUNDS
    check_rows(oracle, w, o, lse, 0, 100, [0, 5, 79])
    check_rows(oracle, w, o, lse, 80, 300, [20, 21, 100, 219])


def test_varlen_sequence_past_the_token_count(oracle):
    """cu_seqlens ends at 400 but only 300 tokens exist: the sequence that would run past
    them is skipped (nothing read or written), the first is exact."""
    w = inputs.varlen([300], 4, 2, 128, 5203, torch.bfloat16)
    o, lse, st = run_varlen(w, [0, 100, 400], 300, 300, 4)
    assert st == A.ATTN_ERR_DEVICE_BOUNDS
    check_rows(oracle, w, o, lse, 0, 100, range(100))
    assert untouched(o, lse, 100, 300)


def test_varlen_cu_seqlens_short_of_the_token_count(oracle):
    """cu_seqlens ends at 250 of 300 tokens: rows 250..299 belong to no sequence and stay
    unwritten; the error is recorded; both sequences are exact."""
    w = inputs.varlen([300], 4, 2, 128, 5204, torch.bfloat16)
    o, lse, st = run_varlen(w, [0, 100, 250], 300, 150, 4)
    assert st == A.ATTN_ERR_DEVICE_BOUNDS
    check_rows(oracle, w, o, lse, 0, 100, range(100))
    check_rows(oracle, w, o, lse, 100, 250, range(150))
    assert untouched(o, lse, 250, 300)


def test_varlen_well_formed_is_not_an_error():
    w = inputs.varlen([0, 130, 1, 0], 4, 2, 64, 5205, torch.bfloat16)
    _, _, st = run_varlen(w, [0, 0, 130, 131, 131], 131, 130, 4)
    assert st == 0


def test_chunk_cu_seqlens_past_the_query_count(oracle):
    """The chunked prefill applies the same packing rules to its queries."""
    ctx, ql = [300, 200], [100, 50]
    w = inputs.chunked(ctx, ql, 4, 2, 128, 5206)
    Tq = 150
    o, obuf = guarded((Tq, 4, 128), torch.bfloat16, SENTINEL_BF16)
    lse, lbuf = guarded((4, Tq), torch.float32, SENTINEL_F32)
    cu = torch.tensor([0, 100, 170], dtype=torch.int32, device="cuda")   # 170 > 150 queries
    A.attn_fwd_chunked_paged(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(),
                             w.page_table.cuda(), w.seq_lens.cuda(), cu, 100, True, w.scale,
                             o=o, lse=lse)
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BOUNDS
    assert_guards_intact(obuf, SENTINEL_BF16)
    assert_guards_intact(lbuf, SENTINEL_F32)
    rows = np.array([(i, h) for h in range(4) for i in range(100)], np.int32)  # (token, head)
    o_ref, l_ref = oracle.chunk_paged_rows(f32(w.q), f32(w.k_cache), f32(w.v_cache),
                                           w.page_table.numpy(), w.seq_lens.numpy(),
                                           w.cu_seqlens_q.numpy(), True, w.scale, rows=rows)
    og = f32(o)[rows[:, 0], rows[:, 1]]
    lg = f32(lse)[rows[:, 1], rows[:, 0]]
    assert_close(errors(og, o_ref, lg, l_ref))
    assert untouched(o, lse, 100, 150)


# ---------------------------------------------------------------- output alignment

@pytest.mark.parametrize("d", [64, 128])
def test_prefill_output_at_a_16_byte_offset(d):
    """The prefill writes O rows with 32-byte stores when O is 32-byte aligned and with
    16-byte stores otherwise (the interface asks for 16-byte alignment).  An O that
    starts 16 bytes past a 32-byte boundary gets the same values, and its guard bands
    stay untouched."""
    w = inputs.dense(2, 300, 4, 2, d, 5401)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o_ref, lse_ref = A.attn_fwd(q, k, v, True, w.scale)
    n = q.numel()
    buf = torch.full((PAD + 8 + n + PAD,), SENTINEL_BF16, dtype=torch.bfloat16, device="cuda")
    o = buf[PAD + 8:PAD + 8 + n].view(q.shape)           # 16 bytes past a 32-byte boundary
    assert o.data_ptr() % 32 == 16
    o2, lse2 = A.attn_fwd(q, k, v, True, w.scale, o=o)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    assert torch.equal(o2, o_ref) and torch.equal(lse2, lse_ref)
    assert bool((buf[:PAD + 8].float() == SENTINEL_BF16).all())
    assert bool((buf[PAD + 8 + n:].float() == SENTINEL_BF16).all())
