"""Pins for the oracle's INT8 cache decode (yapayzekasozluk.tr "attention" tag page,
entry "KV Cache": a cache kept in INT8/FP8 takes 2-4x less memory).  The byte values
are checked against numpy's int8 view of every byte (a library routine); the INT8
decode is checked against the bf16 paged decode entry point on values both hold
exactly, and against the FP8 decode on values both byte formats hold exactly.
"""
import numpy as np
import torch

from attn_fwd_07_b300 import inputs


def test_int8_values_match_numpy_for_every_byte(oracle):
    """All 256 bytes against numpy's two's complement int8 view.  Catches: an unsigned
    reading, an off-by-256 on the negative half."""
    ref = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    got = np.array([oracle.int8_value(b) for b in range(256)])
    np.testing.assert_array_equal(got, ref)
    assert oracle.int8_value(0x80) == -128.0 and oracle.int8_value(0x7F) == 127.0


def test_int8_decode_equals_bf16_decode_on_the_same_values(oracle):
    """With unit scales, the INT8 decode of a cache equals the bf16 paged decode of the
    same integers (every int8 is exact in bf16).  Catches: wrong page lookup, wrong head
    map, wrong byte order."""
    p = inputs.paged_int8([1, 16, 17, 90, 200], 8, 2, 32, 41)
    one = np.ones(2, np.float32)
    o8, l8 = oracle.decode_paged_int8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                      one, one, p.page_table.numpy(), p.seq_lens.numpy(),
                                      p.scale * 0.05)
    kb, vb = (t.float().numpy() for t in (p.k_cache, p.v_cache))
    ob, lb = oracle.decode_paged(p.q.float().numpy(), kb, vb, p.page_table.numpy(),
                                 p.seq_lens.numpy(), p.scale * 0.05)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)


def test_int8_scales_act_per_head(oracle):
    """k_scale[g] = 2^a multiplies head g's keys and v_scale[g] = 2^b its values (powers
    of two keep the float twin exact): equal to the bf16 decode of the scaled values.
    Catches: a scale applied to the wrong head or the wrong tensor."""
    p = inputs.paged_int8([33, 64, 100], 8, 2, 16, 42)
    ks = np.array([2.0 ** -7, 2.0 ** -4], np.float32)
    vs = np.array([2.0 ** -5, 2.0 ** -8], np.float32)
    o8, l8 = oracle.decode_paged_int8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                      ks, vs, p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    kf = p.k_cache.float().numpy() * ks.reshape(1, 1, 2, 1)
    vf = p.v_cache.float().numpy() * vs.reshape(1, 1, 2, 1)
    ob, lb = oracle.decode_paged(p.q.float().numpy(), kf, vf, p.page_table.numpy(),
                                 p.seq_lens.numpy(), p.scale)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)


def test_int8_decode_equals_fp8_decode_on_small_integers(oracle):
    """Integers -16 .. 16 are exact in both byte formats: the same cache written as INT8
    and as E4M3 bytes decodes to the same result.  Catches: either format's value rule
    applied to the other's bytes."""
    p = inputs.paged_int8([7, 40, 129], 8, 4, 32, 43)
    k8 = torch.clamp(p.k_cache, -16, 16)
    v8 = torch.clamp(p.v_cache, -16, 16)
    kf8, vf8 = (t.float().to(torch.float8_e4m3fn).view(torch.uint8) for t in (k8, v8))
    ks = np.full(4, 0.125, np.float32)
    vs = np.full(4, 0.25, np.float32)
    args = (p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    oi, li = oracle.decode_paged_int8(p.q.float().numpy(), k8.numpy(), v8.numpy(), ks, vs, *args)
    of, lf = oracle.decode_paged_fp8(p.q.float().numpy(), kf8.numpy(), vf8.numpy(), ks, vs, *args)
    np.testing.assert_array_equal(oi, of)
    np.testing.assert_array_equal(li, lf)


def test_int8_empty_sequence(oracle):
    p = inputs.paged_int8([0, 5], 2, 1, 16, 44, max_pages=1)
    o, l = oracle.decode_paged_int8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                    p.k_scale.numpy(), p.v_scale.numpy(), p.page_table.numpy(),
                                    p.seq_lens.numpy(), p.scale)
    assert (o[0] == 0).all() and np.isneginf(l[0]).all()
