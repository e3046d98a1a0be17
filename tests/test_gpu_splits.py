"""The paged decode at controlled split counts (GPU).

The decode cuts the pages of all sequences into equal ranges, one per CTA, attends
each range on its own and merges each sequence's pieces by their log-sum-exps: the
rescaling rule of "Donanıma Duyarlı Algoritma Tasarımı: FlashAttention"
(fatihsoysal.com), section "Online Softmax Prensibi", applied to whole key ranges.
The result must not depend on the cut.  The library's own launch always uses one
or two CTAs per SM; the test hook attn_testing_decode_paged_ctas (include/
attn07_testing.h) sets the count, so that one sequence is attended whole (1 CTA),
split in two, split at odd places (7), in many small pieces (64, #SM, 2 x #SM, more
CTAs than some sequences have pages).
"""
import ctypes

import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hook():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = A.load_library()
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn = lib.attn_testing_decode_paged_ctas
    fn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, P, SZ, I, P]
    fn.restype = ctypes.c_int
    assert A.attn_get_device_status() == 0
    return fn


def f32(t):
    return t.float().cpu().numpy()


def run(fn, w, dev, ctas):
    q, kc, vc, pt, sl = dev
    B, Hq, d = q.shape
    P_, ps, Hkv, _ = kc.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = A.attn_decode_workspace_size(B, Hq, d, pt.shape[1], ps)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = fn(p(q), p(kc), p(vc), p(pt), p(sl), p(o), p(lse), B, Hq, Hkv, d, ps, P_, pt.shape[1],
            w.scale, p(ws), need, ctas, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, A.attn_status_string(rc)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    return o, lse


def test_split_counts_match_the_oracle_and_repeat_bitwise(hook, oracle):
    lens = [1, 15, 16, 17, 3000, 1023, 700, 0, 4096, 33]
    w = inputs.paged(lens, 32, 8, 128, 5300, page_size=16)
    dev = [t.cuda() for t in (w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    o_ref, lse_ref = oracle.decode_paged(f32(w.q), f32(w.k_cache), f32(w.v_cache),
                                         w.page_table.numpy(), w.seq_lens.numpy(), w.scale)
    outs = {}
    for ctas in (1, 2, 7, 64, sms, 2 * sms):
        o1, l1 = run(hook, w, dev, ctas)
        o2, l2 = run(hook, w, dev, ctas)
        assert torch.equal(o1, o2) and torch.equal(l1, l2), ctas
        assert_close(errors(f32(o1), o_ref, f32(l1), lse_ref), ctas)
        outs[ctas] = (o1, l1)
    # one CTA attends each sequence whole; every other count splits some of them, and
    # the merged results stay within rounding of it
    o1, l1 = outs[1]
    for ctas, (o, l) in outs.items():
        assert float((o.float() - o1.float()).abs().max()) <= 2e-2, ctas
        empty = torch.isneginf(l) & torch.isneginf(l1)      # the 0-token sequence
        assert float(torch.where(empty, 0.0, l - l1).abs().max()) <= 1e-3, ctas
    # the library's own launch is one of these counts (one CTA per SM for a bf16 cache)
    od, ld = A.attn_decode_paged(*dev, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(od, outs[sms][0]) and torch.equal(ld, outs[sms][1])


def test_split_count_outside_the_workspace_is_refused(hook):
    w = inputs.paged([100], 8, 2, 64, 5301, page_size=16)
    dev = [t.cuda() for t in (w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens)]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q, kc, vc, pt, sl = dev
    need = A.attn_decode_workspace_size(1, 8, 64, pt.shape[1], 16)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    for ctas, want in ((0, A.ATTN_ERR_INVALID_ARG), (2 * sms + 1, A.ATTN_ERR_UNSUPPORTED)):
        rc = hook(p(q), p(kc), p(vc), p(pt), p(sl), p(o), None, 1, 8, 2, 64, 16, kc.shape[0],
                  pt.shape[1], w.scale, p(ws), need, ctas, None)
        assert rc == want, ctas
