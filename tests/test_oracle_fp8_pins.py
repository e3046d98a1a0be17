"""Pins for the oracle's FP8 E4M3 cache decode (yapayzekasozluk.tr "attention" tag
page, entry "KV Cache": a cache kept in INT8/FP8 takes 2-4x less memory).  The
E4M3 byte values are checked against torch's float8_e4m3fn conversion (a
library routine) and hand-worked bit patterns; the FP8 decode is checked
against the bf16 paged decode entry point on values both formats hold exactly.
"""
import numpy as np
import pytest
import torch

from attn_fwd_07_b300 import inputs


def test_e4m3_values_match_torch_for_every_byte(oracle):
    """All 256 bytes against torch's float8_e4m3fn -> float32 conversion.  Catches: a
    wrong bias, a wrong subnormal rule, a sign error."""
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_value(b) for b in range(256)])
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.isnan(got[nan]).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("byte,value", [
    (0x38, 1.0), (0x7E, 448.0), (0x01, 2.0 ** -9), (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9),
    (0xC0, -2.0), (0x3C, 1.5), (0x00, 0.0),
])
def test_e4m3_hand_values(oracle, byte, value):
    """Bit patterns worked by hand: 0x38 = 0 0111 000 = 2^(7-7); 0x7e = 0 1111 110 =
    1.75 * 2^8 (largest); 0x01 = 1/8 * 2^-6 (smallest subnormal); 0x08 = 2^-6 (smallest
    normal); 0xc0 = -2."""
    assert oracle.e4m3_value(byte) == value


def _bf16_twin(p):
    """The FP8 cache's values (unit scale) as bf16 tensors: every E4M3 value is exact in
    bf16, so both oracle entry points see the same numbers."""
    kv = [t.view(torch.float8_e4m3fn).to(torch.bfloat16) for t in (p.k_cache, p.v_cache)]
    return kv


def test_fp8_decode_equals_bf16_decode_on_the_same_values(oracle):
    """With unit scales, the FP8 decode of a cache equals the bf16 paged decode of the
    same values.  Catches: wrong page lookup, wrong head map, wrong byte order."""
    p = inputs.paged_fp8([1, 16, 17, 90, 200], 8, 2, 32, 31)
    one = np.ones(2, np.float32)
    o8, l8 = oracle.decode_paged_fp8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                     one, one, p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    kb, vb = _bf16_twin(p)
    ob, lb = oracle.decode_paged(p.q.float().numpy(), kb.float().numpy(), vb.float().numpy(),
                                 p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)


def test_fp8_scales_act_per_head(oracle):
    """k_scale[g] = 2^a multiplies head g's keys and v_scale[g] = 2^b its values
    (powers of two keep the bf16 twin exact): equal to the bf16 decode of the scaled
    values.  Catches: a scale applied to the wrong head or the wrong tensor."""
    p = inputs.paged_fp8([33, 64, 100], 8, 2, 16, 32)
    ks = np.array([0.5, 4.0], np.float32)
    vs = np.array([0.25, 2.0], np.float32)
    o8, l8 = oracle.decode_paged_fp8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                     ks, vs, p.page_table.numpy(), p.seq_lens.numpy(), p.scale)
    kb, vb = _bf16_twin(p)
    kf = kb.float().numpy() * ks.reshape(1, 1, 2, 1)
    vf = vb.float().numpy() * vs.reshape(1, 1, 2, 1)
    ob, lb = oracle.decode_paged(p.q.float().numpy(), kf, vf, p.page_table.numpy(),
                                 p.seq_lens.numpy(), p.scale)
    np.testing.assert_allclose(o8, ob, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l8, lb, rtol=0, atol=1e-12)


def test_fp8_empty_sequence(oracle):
    p = inputs.paged_fp8([0, 5], 2, 1, 16, 33, max_pages=1)
    o, l = oracle.decode_paged_fp8(p.q.float().numpy(), p.k_cache.numpy(), p.v_cache.numpy(),
                                   p.k_scale.numpy(), p.v_scale.numpy(), p.page_table.numpy(),
                                   p.seq_lens.numpy(), p.scale)
    assert (o[0] == 0).all() and np.isneginf(l[0]).all()
