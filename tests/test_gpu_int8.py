"""GPU parity for the decode against an INT8 paged cache (attn_decode_paged_int8)
against the fp64 oracle on the same bytes and scales.  Ragged lengths, empty
sequences, group sizes 1-8, every byte value (-128 included), a bad page id, and the
64-sequence workload on sampled sequences.  Tolerances are in tests/parity.py."""
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


def run(p):
    return A.attn_decode_paged_int8(*(t.cuda() for t in (p.q, p.k_cache, p.v_cache, p.k_scale,
                                                         p.v_scale, p.page_table, p.seq_lens)),
                                   p.scale)


def ref(oracle, p, seqs=None):
    return oracle.decode_paged_int8(f32(p.q), p.k_cache.numpy(), p.v_cache.numpy(),
                                   p.k_scale.numpy(), p.v_scale.numpy(), p.page_table.numpy(),
                                   p.seq_lens.numpy(), p.scale, seqs=seqs)


@pytest.mark.parametrize("lens,Hq,Hkv", [
    ([1, 15, 16, 17, 1023], 32, 8), ([0, 5, 300, 2048], 8, 8), ([4096, 1, 777], 16, 2),
    ([129, 64, 3000], 8, 1), ([5000, 40], 32, 4),
])
def test_int8_decode_small(oracle, lens, Hq, Hkv):
    p = inputs.paged_int8(lens, Hq, Hkv, 128, 6000 + len(lens) + Hq + Hkv)
    o, lse = run(p)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = ref(oracle, p)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), (lens, Hq, Hkv))


def test_int8_decode_large_scores(oracle):
    """Queries scaled so that scores spread widely (running-maximum rescaling on
    most pages); V scale small so |O| stays in the tolerance's range."""
    p = inputs.paged_int8([700, 3000], 32, 8, 128, 6100)
    p.q = (p.q.float() * 8.0).to(torch.bfloat16)
    p.v_scale = p.v_scale * 0.25
    o, lse = run(p)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = ref(oracle, p)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), "large scores")


def test_int8_every_byte_value(oracle):
    """The cache's bytes run through all 256 values (-128 .. 127, each token row a
    different rotation), so every byte takes the widening to f16; small scales keep the
    scores and |O| in the tolerance's range."""
    p = inputs.paged_int8([300, 77], 16, 4, 128, 6400)
    P_, ps, Hkv, d = p.k_cache.shape
    idx = torch.arange(P_ * ps * Hkv * d, dtype=torch.int64).view(P_, ps, Hkv, d)
    p.k_cache = ((idx * 7 + idx // d) % 256 - 128).to(torch.int8)
    p.v_cache = ((idx * 13 + 3 * (idx // d)) % 256 - 128).to(torch.int8)
    p.k_scale = torch.full((Hkv,), 1.0 / 512, dtype=torch.float32)
    p.v_scale = torch.full((Hkv,), 1.0 / 128, dtype=torch.float32)
    assert int(p.k_cache.min()) == -128 and int(p.v_cache.max()) == 127
    o, lse = run(p)
    torch.cuda.synchronize()
    check_status()
    o_ref, lse_ref = ref(oracle, p)
    assert_close(errors(f32(o), o_ref, f32(lse), lse_ref), "every byte")


def test_int8_bad_page_id_is_reported_not_read(oracle):
    p = inputs.paged_int8([40, 40], 8, 8, 128, 6200)
    pt = p.page_table.clone()
    pt[1, 1] = 10 ** 6
    o, lse = A.attn_decode_paged_int8(*(t.cuda() for t in (p.q, p.k_cache, p.v_cache, p.k_scale,
                                                           p.v_scale, pt, p.seq_lens)), p.scale)
    torch.cuda.synchronize()
    assert A.attn_get_device_status() == A.ATTN_ERR_DEVICE_BOUNDS
    # sequence 0 is untouched by the bad entry
    o_ref, lse_ref = ref(oracle, p, seqs=np.array([0], np.int32))
    assert_close(errors(f32(o)[:1], o_ref, f32(lse)[:1], lse_ref), "seq 0")


def test_int8_rejects_other_head_dims():
    p = inputs.paged_int8([16], 2, 2, 64, 6300)
    with pytest.raises(A.AttnError):
        run(p)


def test_workload_decode_int8_sampled(oracle):
    """B=64, lengths U[1024, 32768], Hq=32 Hkv=8 d=128, INT8 cache (as the benchmark
    runs it), 8 sequences checked against the oracle."""
    w = inputs.make("decode_paged_int8_b64")
    o, lse = run(w)
    torch.cuda.synchronize()
    check_status()
    seqs = np.array([0, 7, 13, 29, 36, 44, 58, 63], np.int32)
    o_ref, lse_ref = ref(oracle, w, seqs=seqs)
    assert_close(errors(f32(o)[seqs], o_ref, f32(lse)[seqs], lse_ref), "decode_paged_int8_b64")
