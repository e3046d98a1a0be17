"""GPU parity for sliding-window prefill (attn_fwd_window) against the fp64
oracle's window rows, on the same seeded inputs.  Windows on either side,
symmetric windows as the sliding-window glossary entry describes them, zero
windows, windows wider than the sequence, both CTA pairings (GQA head pairs and
row-tile pairs), ragged tails, and the 8192-token workload on sampled rows.
Tolerances are in tests/parity.py."""
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


WINDOW_CASES = [
    # B, N, Hq, Hkv, d, wl, wr
    (1, 1, 1, 1, 128, 0, 0), (1, 300, 2, 1, 128, 0, 0), (1, 300, 4, 2, 128, 5, 0),
    (1, 513, 2, 2, 128, 128, 0), (2, 700, 4, 1, 128, 100, 100), (1, 1000, 2, 1, 128, 200, -1),
    (1, 777, 2, 2, 64, -1, 37), (1, 640, 8, 2, 128, 1000, 1000), (1, 1024, 2, 2, 128, 255, 129),
    (3, 385, 6, 3, 64, 64, 64), (1, 900, 1, 1, 128, 300, 0), (1, 256, 4, 4, 64, 0, 127),
]


@pytest.mark.parametrize("B,N,Hq,Hkv,d,wl,wr", WINDOW_CASES)
def test_window_small(oracle, B, N, Hq, Hkv, d, wl, wr):
    seed = 3000 + B * 7 + N + Hq * 5 + d + wl + 2 * wr
    w = inputs.dense(B, N, Hq, Hkv, d, seed, torch.bfloat16)
    o, lse = A.attn_fwd_window(w.q.cuda(), w.k.cuda(), w.v.cuda(), wl, wr, w.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.attn_window(f32(w.q), f32(w.k), f32(w.v), wl, wr, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (B, N, Hq, Hkv, d, wl, wr))


@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 3)])
def test_unbounded_windows_equal_causal_and_full(Hq, Hkv):
    """(-1, 0) is causal and (-1, -1) full attention: bitwise the same kernel work as
    attn_fwd (same tiles, same order)."""
    w = inputs.dense(2, 531, Hq, Hkv, 128, 91, torch.bfloat16)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    for wl, wr, causal in ((-1, 0, True), (-1, -1, False)):
        o1, l1 = A.attn_fwd_window(q, k, v, wl, wr, w.scale)
        o2, l2 = A.attn_fwd(q, k, v, causal, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2), (wl, wr)
    check_status()


def test_window_rejects_bad_extents():
    w = inputs.dense(1, 16, 1, 1, 128, 92, torch.bfloat16)
    with pytest.raises(A.AttnError):
        A.attn_fwd_window(w.q.cuda(), w.k.cuda(), w.v.cuda(), -2, 0, w.scale)


def test_workload_swa_n8192_sampled(oracle):
    """B=1 Hq=32 Hkv=8 N=8192 d=128, 2048 keys left and right (as the benchmark runs
    it): every output checked on sampled rows, including both sequence ends."""
    w = inputs.make("swa_n8192_w4096")
    wl, wr = w.window
    o, lse = A.attn_fwd_window(w.q.cuda(), w.k.cuda(), w.v.cuda(), wl, wr, w.scale)
    torch.cuda.synchronize()
    check_status()
    B, N, Hq, d = w.q.shape
    rng = np.random.default_rng(6)
    i = np.concatenate([[0, 1, 2047, 2048, 4095, 6143, 6144, N - 2, N - 1],
                        rng.integers(0, N, 247)])
    h = rng.integers(0, Hq, len(i))
    rows = np.stack([np.zeros_like(i), h, i], 1).astype(np.int32)
    o_ref, lse_ref = oracle.attn_window_rows(f32(w.q), f32(w.k), f32(w.v), rows, wl, wr,
                                             w.scale)
    og = f32(o)[0, i, h]
    lg = f32(lse)[0, h, i]
    assert_close(errors(og, o_ref, lg, lse_ref), "swa_n8192_w4096")


# ---------------------------------------------------------------- windowed paged decode

@pytest.mark.parametrize("lens,window", [
    ([1, 15, 16, 17, 1023], 0), ([1, 15, 16, 17, 1023], 15), ([300, 2048, 4096], 16),
    ([300, 2048, 4096], 1000), ([5000, 33, 700, 12000], 4095), ([40, 41], 100000),
])
def test_decode_window_small(oracle, lens, window):
    p = inputs.paged(lens, 32, 8, 128, 4000 + window % 997 + len(lens), page_size=16)
    o, lse = A.attn_decode_paged_window(*(t.cuda() for t in (p.q, p.k_cache, p.v_cache,
                                                              p.page_table, p.seq_lens)),
                                        window, p.scale)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = oracle.decode_paged_window(*(f32(t) for t in (p.q, p.k_cache, p.v_cache)),
                                                p.page_table.numpy(), p.seq_lens.numpy(),
                                                window, p.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (lens, window))


def test_decode_window_minus_one_is_plain_decode():
    """window = -1 is attn_decode_paged: bitwise the same split plan and results."""
    p = inputs.paged([100, 2000, 5], 16, 4, 128, 4100, page_size=16)
    args = [t.cuda() for t in (p.q, p.k_cache, p.v_cache, p.page_table, p.seq_lens)]
    o1, l1 = A.attn_decode_paged_window(*args, -1, p.scale)
    o2, l2 = A.attn_decode_paged(*args, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    check_status()


def test_decode_window_workload_sampled(oracle):
    """The 64-sequence decode workload with a 4096-token window, on 8 sequences."""
    w = inputs.make("decode_paged_b64")
    o, lse = A.attn_decode_paged_window(*(t.cuda() for t in (w.q, w.k_cache, w.v_cache,
                                                              w.page_table, w.seq_lens)),
                                        4095, w.scale)
    torch.cuda.synchronize()
    check_status()
    seqs = np.array([0, 5, 17, 23, 31, 40, 52, 63], np.int32)
    o_ref, lse_ref = oracle.decode_paged_window(*(f32(t) for t in (w.q, w.k_cache, w.v_cache)),
                                                w.page_table.numpy(), w.seq_lens.numpy(), 4095,
                                                w.scale, seqs=seqs)
    assert_close(errors(f32(o)[seqs], o_ref, f32(lse)[seqs], lse_ref), "decode window 4095")
