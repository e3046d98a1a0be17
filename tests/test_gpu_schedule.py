"""The tensor-core prefill's work scheduling (GPU).

The persistent CTAs take their work items from a counter in device memory, one of
1024 slots taken in turn by the library's launches; the last CTA of a launch sets its
counter back to zero.  Items are (query-tile level, sequence, head pair) blocks; a
block past a packed sequence's end has no work, and the producer that meets one
moves the counter past the following blocks without work in one step.  None of this
may change a result, so these tests compare against the fp64 oracle or against a
launch whose result is already checked:

- many launches in flight on several streams at once give bitwise the result of one
  launch on its own, also after more launches than there are slots (every slot
  reused);
- packed batches where most blocks have no work (one long sequence among many
  short ones, sequences past the counter's first scan of 64 blocks) match the
  oracle, and so does a batch where every block of the top levels is empty.
"""
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


def test_launches_on_many_streams_match_one_launch():
    w = inputs.dense(2, 1500, 8, 2, 128, 5501)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o_ref, lse_ref = A.attn_fwd(q, k, v, True, w.scale)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(6)]
    outs = []
    for rnd in range(24):                      # 144 launches: every counter slot twice over
        st = streams[rnd % len(streams)]
        with torch.cuda.stream(st):
            o = torch.empty_like(q)
            lse = torch.empty_like(lse_ref)
            A.attn_fwd(q, k, v, True, w.scale, o=o, lse=lse, stream=st)
            outs.append((o, lse))
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    for o, lse in outs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_more_launches_than_counter_slots():
    w = inputs.dense(1, 300, 4, 2, 128, 5502)
    q, k, v = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o_ref, lse_ref = A.attn_fwd(q, k, v, True, w.scale)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(4)]
    bufs = [(torch.empty_like(q), torch.empty_like(lse_ref)) for _ in streams]
    for i in range(1100):                      # past the 1024 slots
        st = streams[i % len(streams)]
        o, lse = bufs[i % len(streams)]
        with torch.cuda.stream(st):
            A.attn_fwd(q, k, v, True, w.scale, o=o, lse=lse, stream=st)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    for o, lse in bufs:
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("lens", [
    [4000] + [1] * 70,                  # one long sequence, 70 one-token ones
    [1] * 40 + [2500] + [3] * 40,       # the long one in the middle
    [129] * 90 + [1800],                # long one last: many empty blocks before it
])
def test_varlen_mostly_empty_blocks(oracle, lens):
    Hq, Hkv, d = 4, 2, 128
    # (values at half scale: rows with one to three keys give |O| near the V values
    # themselves, where a bf16 ulp approaches the tolerance)
    w = inputs.varlen(lens, Hq, Hkv, d, 5600 + len(lens), torch.bfloat16, factor=0.5)
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               max(lens), True, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_varlen(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(),
                                        True, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), lens[:3])


def test_varlen_max_seqlen_above_every_sequence(oracle):
    """max_seqlen sets the launch's query-tile levels; with every sequence much
    shorter, all blocks of the top levels are empty and are skipped."""
    lens = [200, 37, 128, 1]
    Hq, Hkv, d = 8, 4, 64
    w = inputs.varlen(lens, Hq, Hkv, d, 5700, torch.bfloat16, factor=0.5)
    o, lse = A.attn_fwd_varlen(w.q.cuda(), w.k.cuda(), w.v.cuda(), w.cu_seqlens.cuda(),
                               8192, True, w.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == 0
    o_ref, lse_ref = oracle.attn_varlen(f32(w.q), f32(w.k), f32(w.v), w.cu_seqlens.numpy(),
                                        True, w.scale)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), "max_seqlen 8192")
