"""Every output element of the three large workloads against the fp64 oracle (GPU).

The sampled tests in test_gpu_parity.py are the fast tier; these compare all of O
and LSE, in the launch configuration the benchmark times (the same entry points on
the same seeded inputs), and report per workload the largest and mean error, the
worst row and a histogram of |dO| (printed at the end of the run, and written as
JSON with --parity-report PATH).  The oracle needs about a minute for the
16384-token causal prefill and about as long for the packed batch on 16 threads.
"""
import numpy as np
import pytest
import torch

import attn_fwd_07_b300 as A
from attn_fwd_07_b300 import inputs
from parity import assert_close, full_report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    A.load_library()
    assert A.attn_get_device_status() == 0


def f32(t):
    return t.float().cpu().numpy()


def test_full_gqa_causal_n16384(oracle):
    """B=1 Hq=32 Hkv=8 N=16384 d=128 causal: all 67 M output values, 524 288 LSEs."""
    w = inputs.make("gqa_causal_n16384")
    o, lse = A.attn_fwd(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.causal, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(f32(w.q), f32(w.k), f32(w.v), w.causal, w.scale)
    # O is [B, N, Hq, d]: a row is (b, token, head)
    e, _ = full_report("gqa_causal_n16384", f32(o), o_ref, f32(lse), lse_ref, (0, 1, 2))
    assert_close(e)


def test_full_varlen_causal_8seq(oracle):
    """8 packed sequences, lengths U[512, 8192], Hq=32 Hkv=8 d=128 causal: every row."""
    w = inputs.make("varlen_causal_8seq")
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               int(w.lens.max()), True, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_varlen(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(),
                                        True, w.scale)
    # O is [T, Hq, d]: a row is (token, head)
    e, _ = full_report("varlen_causal_8seq", f32(o), o_ref, f32(lse), lse_ref, (0, 1))
    assert_close(e)


def test_full_decode_paged_b64(oracle):
    """B=64 decode against the 1.15 M-token paged cache: all 64 sequences, every head.
    The oracle takes the sequences eight at a time, each group's pages gathered into a
    compact cache (the page table renumbered accordingly)."""
    w = inputs.make("decode_paged_b64")
    dev = [t.cuda() for t in (w.q, w.k_cache, w.v_cache, w.page_table, w.seq_lens)]
    o, lse = A.attn_decode_paged(*dev, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    lens = w.seq_lens.numpy()
    ps = w.page_size
    B = len(lens)
    o_ref = np.zeros((B,) + tuple(w.q.shape[1:]), np.float64)
    lse_ref = np.zeros((B, w.q.shape[1]), np.float64)
    for g0 in range(0, B, 8):
        seqs = list(range(g0, min(B, g0 + 8)))
        pages = [w.page_table[b, :(int(lens[b]) + ps - 1) // ps].numpy() for b in seqs]
        idx = torch.from_numpy(np.concatenate(pages)).long()
        kc, vc = f32(w.k_cache[idx]), f32(w.v_cache[idx])
        pt = np.full((len(seqs), max(len(p) for p in pages)), -1, np.int32)
        off = 0
        for r, p in enumerate(pages):
            pt[r, :len(p)] = np.arange(off, off + len(p))
            off += len(p)
        o_ref[seqs], lse_ref[seqs] = oracle.decode_paged(f32(w.q)[seqs], kc, vc, pt,
                                                         lens[seqs], w.scale)
    # O is [B, Hq, d]: a row is (sequence, head)
    e, _ = full_report("decode_paged_b64", f32(o), o_ref, f32(lse), lse_ref, (0, 1))
    assert_close(e)
